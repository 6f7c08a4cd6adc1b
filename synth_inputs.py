"""Seeded synthetic inputs for the Q4 verify matmul.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It holds no arithmetic of the method: it draws random numbers, rounds
them to bf16 (round to nearest even, the input recipe) and lays the drawn
values out in the packed weight format so that both sides read the same bytes.

Input recipe (every config):
  * nibbles q uniform in 0..15 (uniform random bytes: both nibbles uniform and
    independent);
  * scale  = bf16_RNE(|N(0,1)| * 0.01), one per (row n, group of 64 inputs);
  * bias   = bf16_RNE(-8 * scale + N(0, 0.001)), computed from the rounded scale;
  * x      = bf16_RNE(N(0,1)), M rows of K inputs.

Packed layout (planar, row-major; total N*K/16*9 bytes):
  [nibbles: N rows x K/2 bytes; byte j of a row holds inputs 2j (bits 0-3) and
   2j+1 (bits 4-7)]
  [scales:  N rows x K/64 bf16, little-endian]
  [biases:  N rows x K/64 bf16, little-endian]
"""
from __future__ import annotations

import torch

GROUP = 64


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> int16 tensor holding the same bit patterns."""
    return t.contiguous().view(torch.int16)


def make_weights(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """Packed uint8 buffer of exactly N*K/16*9 bytes on ``device``."""
    if K % GROUP != 0 or N < 1:
        raise ValueError("K must be a multiple of 64 and N >= 1")
    G = K // GROUP
    g = _gen(seed, device)
    nib = torch.randint(0, 256, (N * (K // 2),), generator=g, device=device, dtype=torch.int32)
    nib = nib.to(torch.uint8)
    scale = (torch.randn((N, G), generator=g, device=device, dtype=torch.float32).abs() * 0.01)
    scale = scale.to(torch.bfloat16)
    noise = torch.randn((N, G), generator=g, device=device, dtype=torch.float32) * 0.001
    bias = (scale.to(torch.float32) * -8.0 + noise).to(torch.bfloat16)
    return torch.cat([nib, scale.contiguous().view(torch.uint8).reshape(-1),
                      bias.contiguous().view(torch.uint8).reshape(-1)])


def make_x(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [M, K] activations, N(0,1) rounded to nearest even."""
    g = _gen(seed, device)
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def pack_planes(nibbles: torch.Tensor, scales_bf16: torch.Tensor, biases_bf16: torch.Tensor) -> torch.Tensor:
    """Concatenate already-formed planes (uint8 [N, K/2], bf16 [N, K/64] x 2)."""
    return torch.cat([nibbles.contiguous().reshape(-1).to(torch.uint8),
                      scales_bf16.contiguous().view(torch.uint8).reshape(-1),
                      biases_bf16.contiguous().view(torch.uint8).reshape(-1)])


# Seeds, fixed per workload so that every run draws the same inputs.  Workloads
# are numbered 1..5 in the order: tiny, attention projection, MLP/GDN shapes,
# LM head, full chained pass.
def w_seed(workload: int, tensor_index: int = 0) -> int:
    return tensor_index if workload == 1 else 1000 * workload + tensor_index


def x_seed(workload: int) -> int:
    return 1 if workload == 1 else 1000 * workload + 999


# Named shapes of the 27B-class hybrid model (hidden 5120, intermediate 17408,
# attention projection 14336 = 6144 + 1024 + 1024 + 6144, GDN projection 16640,
# vocabulary 248320), taken from the "Splash engine" page's model struct.
HIDDEN = 5120
INTERMEDIATE = 17408
VOCAB = 248320
ATTN_IN = 14336
GDN_IN = 16640
ATTN_OUT_IN = 6144      # attention output projection input width (24 heads x 256)
GDN_OUT_IN = 6144       # GDN output projection input width (48 value heads x 128)

SHAPES = {
    "tiny": (256, 512),
    "attn_in": (ATTN_IN, HIDDEN),
    "gate_up": (2 * INTERMEDIATE, HIDDEN),
    "down": (HIDDEN, INTERMEDIATE),
    "gdn_in": (GDN_IN, HIDDEN),
    "gdn_out": (HIDDEN, GDN_OUT_IN),
    "attn_out": (HIDDEN, ATTN_OUT_IN),
    "lm_head": (VOCAB, HIDDEN),
}


def full_pass_spec():
    """(N, K, glue) of every linear of the 27B-shaped verify pass, in order: 64
    layers (attention when i % 4 == 3, Gated DeltaNet otherwise, the page's
    fullAttentionPeriod of 4), each [in-proj, out-proj, gate/up, down], then the
    LM head twice (target verify, draft readout).  glue: 1 = first K columns,
    2 = SwiGLU halves, 0 = end of the step (the library's glue kinds)."""
    spec = []
    for i in range(64):
        n_in = ATTN_IN if i % 4 == 3 else GDN_IN
        spec += [(n_in, HIDDEN, 1), (HIDDEN, ATTN_OUT_IN, 1), (2 * INTERMEDIATE, HIDDEN, 2), (HIDDEN, INTERMEDIATE, 1)]
    spec += [(VOCAB, HIDDEN, 1), (VOCAB, HIDDEN, 0)]
    return spec


# ------------------------------------------------------------ draft selector
# Edge-score inputs: two bf16 codebooks [VOCAB, 256], each entry N(0,1) * 0.05
# rounded to nearest even; per (lane, position) row a hidden projection of 256
# N(0,1) fp32 values; the 16 candidates of a position are 16 distinct token ids
# drawn uniformly; the predecessors of position p > 0 are the candidates of
# position p - 1, and those of position 0 are the lane's anchor token, repeated.
EDGE_RANK = 256
EDGE_POSITIONS = 7
EDGE_PAIRS = 16


def make_codebook(V: int, R: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn((V, R), generator=g, device=device, dtype=torch.float32) * 0.05).to(torch.bfloat16)


def make_edge_inputs(lanes: int, V: int, R: int, seed: int, positions: int = EDGE_POSITIONS):
    """(hidden fp32 [rows, R], pred_ids int32 [rows, 16], cand_ids int32 [rows, 16]) on the CPU,
    rows = lanes * positions, row = lane * positions + position."""
    g = _gen(seed, "cpu")
    rows = lanes * positions
    hidden = torch.randn((rows, R), generator=g, dtype=torch.float32)
    cand = torch.empty((rows, EDGE_PAIRS), dtype=torch.int32)
    pred = torch.empty((rows, EDGE_PAIRS), dtype=torch.int32)
    for lane in range(lanes):
        anchor = int(torch.randint(0, V, (1,), generator=g))
        for p in range(positions):
            r = lane * positions + p
            cand[r] = torch.randperm(V, generator=g)[:EDGE_PAIRS].to(torch.int32) if V >= 4 * EDGE_PAIRS else \
                torch.randint(0, V, (EDGE_PAIRS,), generator=g, dtype=torch.int32)
            pred[r] = cand[r - 1] if p > 0 else torch.full((EDGE_PAIRS,), anchor, dtype=torch.int32)
    return hidden, pred, cand
