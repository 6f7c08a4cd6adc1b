"""q4_decode_step and q4_glue on the GPU: the chained verify pass ("Splash
engine" analysis, section "The decode step is one command buffer": every layer of
the step runs in order in one submission).

Teacher-forced checks: each layer's GPU output is compared with the oracle
applied to the GPU's own bf16 input of that layer, and each glue output with the
oracle's glue of the GPU's own y.  The glue rounds once to bf16 from a value it
forms to well below a bf16 ulp, so it may differ from the all-double oracle only
by one ulp and only where the exact value lies at a bf16 rounding tie, within a
stated relative distance of the midpoint (see _check_glue).  The whole step
through q4_decode_step must equal the layer-by-layer run bit for bit."""
import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import oracle
import synth_inputs as si
from parity import check_tolerance, sample_columns, xbits

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _rows_of(W: torch.Tensor, N: int, K: int, rows: np.ndarray) -> torch.Tensor:
    """The packed matrix of the given output rows of W (gathered on W's device, returned on the CPU)."""
    G = K // 64
    idx = torch.as_tensor(rows, device=W.device, dtype=torch.long)
    nib = W[: N * K // 2].view(N, K // 2)[idx]
    sb = W[N * K // 2:].view(torch.bfloat16)
    scales = sb[: N * G].view(N, G)[idx]
    biases = sb[N * G:].view(N, G)[idx]
    return si.pack_planes(nib.cpu(), scales.cpu(), biases.cpu())


def _check_layer(x: torch.Tensor, W: torch.Tensor, N: int, K: int, y: torch.Tensor, cols, what: str):
    """GPU y of one layer against the oracle on the GPU's own input x."""
    if cols is None:
        cols = np.arange(N)
    Wsub = _rows_of(W, N, K, cols).numpy()
    ref, scale = oracle.matmul(xbits(x), Wsub, len(cols), K)
    check_tolerance(y.cpu().numpy()[:, cols], ref, scale, what)


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_glue(y: torch.Tensor, K_next: int, kind: int, x_next: torch.Tensor, what: str):
    """GPU glue output against the oracle's glue of the same fp32 y.  A differing
    element must be one bf16 ulp away and lie at a tie: its value (recomputed here
    in double only to classify the difference) is within `rel` of the midpoint
    between the two candidates.  RMSNORM: rel = 1e-9 (the kernel's scale and each
    output are formed to about 1e-14).  SWIGLU: rel = 2e-6, because the kernel's
    sum of squares is taken over the fp32 values silu(a) * b, each within 9 float
    ulps of exact, so its scale is within about 5e-7 of the all-double one."""
    ref = oracle.glue(y.cpu().numpy(), K_next, kind)
    got = si.bf16_bits(x_next.cpu()).numpy().view(np.uint16)
    diff = got != ref
    if not diff.any():
        return
    d = np.abs(got[diff].astype(np.int32) - ref[diff].astype(np.int32))
    assert int(d.max()) <= 1, f"{what}: glue differs from the oracle by {int(d.max())} ulp"
    yy = y.cpu().numpy().astype(np.float64)
    if kind == q4.GLUE_SWIGLU_RMSNORM:
        a = yy[:, :K_next]
        v = a / (1.0 + np.exp(-a)) * yy[:, K_next:2 * K_next]
    else:
        v = yy[:, :K_next]
    inv = 1.0 / np.sqrt(np.mean(v * v, axis=1, keepdims=True) + 1e-6)
    t = (v * inv)[diff]
    mid = 0.5 * (_bf16_value(got[diff]) + _bf16_value(ref[diff]))
    rel = np.abs(t - mid) / np.maximum(np.abs(t), 1e-300)
    lim = 2e-6 if kind == q4.GLUE_SWIGLU_RMSNORM else 1e-9
    assert np.all(rel <= lim), (f"{what}: {int(np.sum(rel > lim))} of {int(diff.sum())} differing outputs are not "
                                f"at a bf16 tie (max distance {rel.max():.3g})")


def _run_by_layers(layers, x0, checks=True, sample=None, tag=""):
    """The chained pass one kernel at a time; returns the last y."""
    x = x0
    y = None
    for j, (W, N, K, g) in enumerate(layers):
        y = q4.matmul(x, W, N, K)
        if checks:
            cols = None if sample is None else sample_columns(N, sample, seed=N + K + j)
            _check_layer(x, W, N, K, y, cols, f"{tag} layer {j} (N={N} K={K})")
        if j + 1 < len(layers):
            Kn = layers[j + 1][2]
            x = q4.glue(y, Kn, g)
            if checks:
                _check_glue(y, Kn, g, x, f"{tag} glue {j}")
    return y


# RMSNORM up to 6144 inputs: every CTA sums its row alone; beyond, and SWIGLU: a cluster per row
@pytest.mark.parametrize("kind,N_prev,K", [(q4.GLUE_RMSNORM, 640, 576), (q4.GLUE_RMSNORM, 5120, 5120),
                                           (q4.GLUE_RMSNORM, 16640, 6144), (q4.GLUE_RMSNORM, 10240, 8192),
                                           (q4.GLUE_SWIGLU_RMSNORM, 2 * 17408, 17408),
                                           (q4.GLUE_SWIGLU_RMSNORM, 2048, 1024)])
def test_glue_against_oracle(kind, N_prev, K):
    g = torch.Generator(device="cpu").manual_seed(N_prev + K)
    y = (torch.randn((16, N_prev), generator=g) * 3.0).to(torch.float32)
    x = q4.glue(y.cuda(), K, kind)
    q4.device_status()
    _check_glue(y, K, kind, x, f"glue kind {kind} {N_prev}->{K}")


def test_glue_rows_are_independent():
    y = torch.randn((16, 2048), generator=torch.Generator().manual_seed(5)).cuda()
    full = si.bf16_bits(q4.glue(y, 1024, q4.GLUE_SWIGLU_RMSNORM).cpu())
    for m in (0, 7, 15):
        alone = si.bf16_bits(q4.glue(y[m:m + 1].contiguous(), 1024, q4.GLUE_SWIGLU_RMSNORM).cpu())
        assert torch.equal(alone[0], full[m])


def _small_chain(device="cuda"):
    """Five layers: both glue kinds between two tensor-memory matmuls (formed
    inside the matmul kernels; the second from a ragged N = 1100 whose first
    1024 outputs feed the next layer), a K that is not a multiple of 512 (the
    generic kernel: the glue kernel writes its x, then the next matmul's
    records) and a ragged last N."""
    spec = [(2048, 512, q4.GLUE_SWIGLU_RMSNORM), (1100, 1024, q4.GLUE_RMSNORM), (1280, 1024, q4.GLUE_RMSNORM),
            (1024, 576, q4.GLUE_RMSNORM), (300, 1024, q4.GLUE_NONE)]
    return [(si.make_weights(N, K, 900 + i, device=device), N, K, g) for i, (N, K, g) in enumerate(spec)]


@pytest.mark.parametrize("M", [1, 3, 16, 24, 32])
def test_small_chain_teacher_forced(M):
    layers = _small_chain()
    x0 = si.make_x(M, 512, 950 + M, device="cuda")
    y_layers = _run_by_layers(layers, x0, tag=f"M={M}")
    y_step = q4.decode_step(layers, x0)
    q4.device_status()
    assert torch.equal(y_step, y_layers), "q4_decode_step differs from the same kernels run one at a time"


def test_small_chain_rows_independent_of_M():
    layers = _small_chain()
    x32 = si.make_x(32, 512, 960, device="cuda")
    y32 = q4.decode_step(layers, x32).cpu()
    for M in (1, 2, 5, 8, 16, 17, 24):
        yM = q4.decode_step(layers, x32[:M].contiguous()).cpu()
        assert torch.equal(yM, y32[:M]), f"M={M}"


def test_decode_step_repeat_is_deterministic():
    layers = _small_chain()
    x = si.make_x(16, 512, 961, device="cuda")
    first = q4.decode_step(layers, x).cpu()
    ws = torch.empty(q4.decode_step_workspace_bytes(layers, 16), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        assert torch.equal(q4.decode_step(layers, x, workspace=ws).cpu(), first)


def test_decode_step_in_a_cuda_graph():
    """The step captured once and replayed gives the eager result for new inputs."""
    layers = _small_chain()
    x = si.make_x(16, 512, 962, device="cuda")
    ws = torch.empty(q4.decode_step_workspace_bytes(layers, 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((16, 300), dtype=torch.float32, device="cuda")
    q4.decode_step(layers, x, y_last=y, workspace=ws)          # device set-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.decode_step(layers, x, y_last=y, workspace=ws, stream=s)
    for seed in (963, 964):
        x.copy_(si.make_x(16, 512, seed, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        ref = q4.decode_step(layers, x).cpu()
        assert torch.equal(y.cpu(), ref)


def _full_pass_layers(device="cuda"):
    """The 27B-shaped pass: 64 layers (attention when i % 4 == 3, Gated DeltaNet
    otherwise), each [in-proj, out-proj, gate/up, down], then the LM head twice."""
    return [(si.make_weights(N, K, si.w_seed(5, t), device=device), N, K, g)
            for t, (N, K, g) in enumerate(si.full_pass_spec())]


@pytest.mark.slow
def test_full_27b_pass_teacher_forced():
    """Every linear of the 64-layer pass and both LM-head calls, M=16: 512
    sampled output columns per layer against the oracle on the GPU's own
    inputs, every glue against the oracle, and the one-submission step equal to
    the layer-by-layer run bit for bit."""
    layers = _full_pass_layers()
    total = sum(N * K * 9 // 16 for _, N, K, _ in layers)
    assert total == 15_149_629_440
    x0 = si.make_x(16, 5120, si.x_seed(5), device="cuda")
    y_layers = _run_by_layers(layers, x0, sample=512, tag="27B")
    y_step = q4.decode_step(layers, x0)
    q4.device_status()
    assert torch.equal(y_step, y_layers)
