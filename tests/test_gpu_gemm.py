"""GPU: the tcgen05 grouped GEMM (moe_expert_up / moe_expert_down, bf16 layers) and the
tensor-core router, called through the C ABI on hand-built group layouts, against the
fp64 oracle.  Cases grow from one tile to ragged groups so a failure points at its cause.

Bounds: h and y_perm (fp16) elementwise within one fp16 rounding of the exact value plus
1e-4 RMS; logits within fp32-accumulation error (1e-5 relative)."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_04_b300 import build as B
from routing_dispatch_expert_04_b300 import native as N
from parity_helpers import assert_rounded_to, rel_rms_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    B.build()
    N.lib()


def _gen(shape, std, seed, dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device="cuda") * std).to(dtype)


@pytest.fixture(params=[N.GEMM_SINGLE, N.GEMM_PAIR, N.GEMM_SPLIT, N.GEMM_PAIR_T, N.GEMM_MIXED],
                ids=["single", "pair", "split", "pair_t", "mixed"])
def pairing(request):
    """Run the case on the one-CTA kernel, the CTA-pair kernel, the split of the two, the
    transposed pair kernel and the mixed-tile pair kernel."""
    N.set_gemm_pairing(request.param)
    yield request.param
    N.set_gemm_pairing(N.GEMM_AUTO)


CASES = [
    # (name, offsets, Kd (=d for up), N (=F for up))
    ("one_tile", [0, 128], 64, 256),
    ("k_blocks", [0, 128], 512, 256),
    ("multi_tile_ragged_m", [0, 300], 320, 768),
    ("groups_empty_and_single_row", [0, 0, 130, 131, 400, 520], 136, 384),
    ("many_groups", list(np.cumsum([0] + [37 * (i % 5) for i in range(40)])), 256, 512),
    ("pair_tiles_ragged", [0, 600, 600, 856, 1111, 1367], 1024, 512),
    # more tiles than SMs for every plan, ragged groups
    ("many_tiles_ragged", list(np.cumsum([0, 700, 512, 0, 1000, 640, 383, 900, 250])), 512, 2048),
]


@pytest.mark.parametrize("name,offs,Kd,Nn", CASES, ids=[c[0] for c in CASES])
def test_expert_up_gelu_f16(name, offs, Kd, Nn, pairing):
    G = len(offs) - 1
    rows = int(offs[-1])
    rows_cap = rows + 64  # spare rows must stay untouched
    cfg = N.make_config(max(rows, 1), Kd, G, 1, Nn, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    x = _gen((rows_cap, Kd), 1.0, 1, torch.bfloat16)
    w1 = _gen((G, Nn, Kd), Kd ** -0.5, 2, torch.bfloat16)
    h = torch.full((rows_cap, Nn), 7.0, dtype=torch.float16, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    N.expert_up(cfg, x, off_t, G, rows_cap, w1, h, ws)
    assert N.sync_status(ws) == 0
    xn, wn, hn = to_np(x), to_np(w1), h.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            ref = O.gelu(O.linear(xn[lo:hi], wn[g]))
            assert_rounded_to(hn[lo:hi], ref, "f16")
    assert (hn[rows:] == 7.0).all()


@pytest.mark.parametrize("name,offs,Kd,Nn", CASES, ids=[c[0] for c in CASES])
def test_expert_down_f16(name, offs, Kd, Nn, pairing):
    G = len(offs) - 1
    rows = int(offs[-1])
    rows_cap = rows + 64
    cfg = N.make_config(max(rows, 1), Nn, G, 1, Kd, "bf16", -1)  # down: N = d, Kd = F
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    h = _gen((rows_cap, Kd), 0.5, 3, torch.float16)
    w2 = _gen((G, Nn, Kd), Kd ** -0.5, 4, torch.float16)
    y = torch.full((rows_cap, Nn), 7.0, dtype=torch.float16, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    N.expert_down(cfg, h, off_t, G, rows_cap, w2, y, ws)
    assert N.sync_status(ws) == 0
    hn, wn, yn = h.float().cpu().numpy(), w2.float().cpu().numpy(), y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            ref = O.linear(hn[lo:hi], wn[g])
            assert_rounded_to(yn[lo:hi], ref, "f16")
    assert (yn[rows:] == 7.0).all()


@pytest.mark.parametrize("T,E,d,bias", [(300, 8, 256, False), (257, 128, 512, True),
                                        (130, 256, 1024, True), (64, 5, 64, True),
                                        (512, 8, 1024, True), (600, 8, 832, False)])
def test_tensor_core_router(T, E, d, bias):
    """Router logits against the fp64 oracle.  The cases cover one K slice (64, 5, 64),
    4 slices, 8 slices of one k-block each (257, 128, 512), 8 slices of two (130, 256,
    1024 and 512, 8, 1024: two CTAs per SM) and 7 slices whose last one is shorter
    (600, 8, 832: 13 k-blocks in slices of two)."""
    cfg = N.make_config(T, d, E, min(2, E), 64, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    x = _gen((T, d), 1.0, 5, torch.bfloat16)
    wr = _gen((E, d), d ** -0.5, 6, torch.bfloat16)
    b = _gen((E,), 0.5, 7, torch.float32) if bias else None
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    N.route(cfg, x, wr, b, logits, ids, w, ws)
    assert N.sync_status(ws) == 0
    L64, _ = O.router_logits(to_np(x), to_np(wr), None if b is None else to_np(b))
    Lg = to_np(logits)
    assert np.max(np.abs(Lg - L64) / (1.0 + np.abs(L64))) <= 1e-5


def _bf16_values(lo, hi):
    """Every finite bf16 value in [lo, hi], as float32."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (v >= lo) & (v <= hi)]
    return np.unique(v)


def test_gelu_epilogue_accuracy_every_bf16_input(pairing):
    """The GEMM1 epilogue's GELU on every bf16 value in [-16, 16], one value per row: A row r
    is (v_r, 0, ..., 0) and every W1 row is (1, 0, ..., 0), so the accumulator is v_r
    exactly and h[r, n] = fp16(GELU(v_r)).  Bound: half an fp16 ulp of the exact GELU (the
    storage rounding) plus 4e-7 for the evaluation (the approximation of the normal tail
    is within 7.5e-8 of Phi; in fp32 the epilogue's GELU is within 3.4e-7 of the exact)."""
    from scipy.special import erf
    v = _bf16_values(-16.0, 16.0)
    rows, Kd, Nn = len(v), 64, 256
    cfg = N.make_config(rows, Kd, 1, 1, Nn, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    a = torch.zeros((rows, Kd), dtype=torch.bfloat16, device="cuda")
    a[:, 0] = torch.from_numpy(v).to(torch.bfloat16).cuda()
    w = torch.zeros((1, Nn, Kd), dtype=torch.bfloat16, device="cuda")
    w[:, :, 0] = 1.0
    h = torch.zeros((rows, Nn), dtype=torch.float16, device="cuda")
    off = torch.tensor([0, rows], dtype=torch.int32, device="cuda")
    N.expert_up(cfg, a, off, 1, rows, w, h, ws)
    assert N.sync_status(ws) == 0
    hn = h.float().cpu().numpy().astype(np.float64)
    assert (hn == hn[:, :1]).all()
    vd = v.astype(np.float64)
    exact = 0.5 * vd * (1.0 + erf(vd / np.sqrt(2.0)))
    ulp = np.spacing(np.abs(exact).astype(np.float16)).astype(np.float64)
    err = np.abs(hn[:, 0] - exact)
    excess = err - (0.5 * ulp + 4e-7)
    i = int(np.argmax(excess))
    assert excess[i] <= 0, (v[i], hn[i, 0], exact[i])


def test_f16_conversion_exact_and_range_error():
    src = _gen((4096,), 0.05, 8, torch.bfloat16)
    src[7] = 1e-6   # below 2^-17: rounds at 2^-25
    dst = torch.empty(4096, dtype=torch.float16, device="cuda")
    cfg = N.make_config(1, 8, 1, 1, 8, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    N.bf16_to_f16(src, dst, ws)
    assert N.sync_status(ws) == 0
    a, b = src.float().cpu().numpy(), dst.float().cpu().numpy()
    big = np.abs(a) >= 2.0 ** -17
    assert np.array_equal(a[big], b[big])
    assert np.max(np.abs(a - b)) <= 2.0 ** -25
    src[100] = 70000.0
    N.bf16_to_f16(src, dst, ws)
    assert N.sync_status(ws) == 5


@pytest.mark.parametrize("fn", ["up", "down"])
def test_single_and_pair_kernels_agree_bitwise(fn):
    """All kernels multiply the same operands and accumulate the 64-deep k-blocks in the
    same order; their outputs are compared bit for bit."""
    offs = [0, 300, 812, 813, 1400]
    G, rows, Kd, Nn = 4, 1400, 512, 768
    rows_cap = rows + 16
    cfg = N.make_config(rows, Kd if fn == "up" else Nn, G, 1, Nn if fn == "up" else Kd, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    outs = []
    for mode in (N.GEMM_SINGLE, N.GEMM_PAIR, N.GEMM_SPLIT, N.GEMM_PAIR_T, N.GEMM_MIXED):
        N.set_gemm_pairing(mode)
        try:
            if fn == "up":
                a = _gen((rows_cap, Kd), 1.0, 11, torch.bfloat16)
                w = _gen((G, Nn, Kd), Kd ** -0.5, 12, torch.bfloat16)
                out = torch.zeros((rows_cap, Nn), dtype=torch.float16, device="cuda")
                N.expert_up(cfg, a, off_t, G, rows_cap, w, out, ws)
            else:
                a = _gen((rows_cap, Kd), 0.5, 13, torch.float16)
                w = _gen((G, Nn, Kd), Kd ** -0.5, 14, torch.float16)
                out = torch.zeros((rows_cap, Nn), dtype=torch.float16, device="cuda")
                N.expert_down(cfg, a, off_t, G, rows_cap, w, out, ws)
        finally:
            N.set_gemm_pairing(N.GEMM_AUTO)
        assert N.sync_status(ws) == 0
        outs.append(out.cpu())
    for i in range(1, len(outs)):
        assert torch.equal(outs[0], outs[i]), i


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("offs,T,K", [([0, 128], 300, 2), ([0, 0, 130, 131, 400, 520], 700, 3),
                                      ([0, 600, 600, 856, 1111, 1367], 900, 2)])
def test_expert_up_gather(offs, T, K, dtype, pairing):
    """Dispatch fused into the first expert Linear: packed row r is gathered from token
    row src[r] // K of x while the tile loads.  Against the oracle, and bit for bit
    against the same GEMM on rows copied in advance."""
    if dtype == "f32" and pairing not in (N.GEMM_SINGLE,):
        pytest.skip("fp32 layers run on the CUDA cores; pairing does not apply")
    G = len(offs) - 1
    rows = int(offs[-1])
    rows_cap = rows + 32
    Kd, Nn = 192, 512
    cfg = N.make_config(T, Kd, max(G, K), K, Nn, dtype, -1)  # K <= E; G groups are passed
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    hdt = torch.float16 if dtype == "bf16" else torch.float32
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    x = _gen((T, Kd), 1.0, 21, tdt)
    w1 = _gen((G, Nn, Kd), Kd ** -0.5, 22, tdt)
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    src = torch.randint(0, T * K, (rows_cap,), generator=g, device="cuda", dtype=torch.int32)
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    h = torch.full((rows_cap, Nn), 7.0, dtype=hdt, device="cuda")
    N.expert_up_gather(cfg, x, src, off_t, G, rows_cap, w1, h, ws)
    assert N.sync_status(ws) == 0
    xp = x[(src.long() // K)].contiguous()   # the same rows, copied (test input only)
    h2 = torch.full((rows_cap, Nn), 7.0, dtype=hdt, device="cuda")
    N.expert_up(cfg, xp, off_t, G, rows_cap, w1, h2, ws)
    assert N.sync_status(ws) == 0
    assert torch.equal(h[:rows], h2[:rows])
    hn, xn, wn, sn = h.float().cpu().numpy(), to_np(x), to_np(w1), src.cpu().numpy()
    for gi in range(G):
        lo, hi = int(offs[gi]), int(offs[gi + 1])
        if hi > lo:
            ref = O.gelu(O.linear(xn[sn[lo:hi] // K], wn[gi]))
            if dtype == "bf16":
                assert_rounded_to(hn[lo:hi], ref, "f16")
            else:
                assert rel_rms_err(hn[lo:hi], ref) <= 1e-4
    assert (hn[rows:] == 7.0).all()


def test_expert_up_gather_bad_index_reported():
    T, K, G, Kd, Nn = 64, 2, 1, 64, 256
    cfg = N.make_config(T, Kd, K, K, Nn, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    x = _gen((T, Kd), 1.0, 31, torch.bfloat16)
    w1 = _gen((G, Nn, Kd), Kd ** -0.5, 32, torch.bfloat16)
    src = torch.arange(100, dtype=torch.int32, device="cuda")
    src[7] = T * K + 5                       # token T + 2: out of range
    off_t = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    h = torch.empty((100, Nn), dtype=torch.float16, device="cuda")
    N.expert_up_gather(cfg, x, src, off_t, G, 100, w1, h, ws)
    assert N.sync_status(ws) == 5  # MOE_ERR_DEVICE


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_grouped_ffn_through_the_abi(dtype):
    """moe_grouped_ffn (both expert Linears, chained on the device through h) on a ragged
    layout with an empty group, on the default plan, against the oracle's expert FFN:
    h within its storage rounding, y_perm against the oracle applied to the h the GPU
    stored (isolating the second Linear) and within the layer tolerance of the exact
    expert output; rows past the groups untouched; bad arguments rejected before any
    launch."""
    offs = [0, 200, 200, 457, 1000, 1129]
    G, rows, d, F = len(offs) - 1, offs[-1], 256, 512
    rows_cap = rows + 32
    cfg = N.make_config(rows, d, G, 1, F, dtype, -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    hdt = torch.float16 if dtype == "bf16" else torch.float32
    x = _gen((rows_cap, d), 1.0, 11, tdt)
    w1 = _gen((G, F, d), d ** -0.5, 12, tdt)
    w2 = _gen((G, d, F), F ** -0.5, 13, tdt)
    w2k = w2
    if dtype == "bf16":  # the second Linear takes fp16 weights (converted once)
        w2k = torch.empty(w2.shape, dtype=torch.float16, device="cuda")
        N.bf16_to_f16(w2, w2k, ws)
    h = torch.full((rows_cap, F), 7.0, dtype=hdt, device="cuda")
    y = torch.full((rows_cap, d), 7.0, dtype=hdt, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    N.grouped_ffn(cfg, x, off_t, G, rows_cap, w1, w2k, h, y, ws)
    assert N.sync_status(ws) == 0
    xn, w1n, w2n = to_np(x), to_np(w1), to_np(w2)
    hn, yn = h.float().cpu().numpy(), y.float().cpu().numpy()
    sdt = "f16" if dtype == "bf16" else "f32"
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        y_ref, h_ref = O.expert_ffn(xn[lo:hi], w1n[g], w2n[g])
        assert_rounded_to(hn[lo:hi], h_ref, sdt)
        assert_rounded_to(yn[lo:hi], O.linear(hn[lo:hi], w2n[g]), sdt)
        assert rel_rms_err(yn[lo:hi], y_ref) <= (2e-2 if dtype == "bf16" else 1e-4)
    assert (hn[rows:] == 7.0).all() and (yn[rows:] == 7.0).all()
    with pytest.raises(N.MoeError):
        N.grouped_ffn(cfg, x, off_t, 0, rows_cap, w1, w2k, h, y, ws)   # no groups
    with pytest.raises(N.MoeError):
        N.grouped_ffn(cfg, x, off_t, G, rows_cap, w1, None, h, y, ws)  # no W2
    with pytest.raises(N.MoeError):
        N.grouped_ffn(cfg, x.view(-1)[1:], off_t, G, rows_cap, w1, w2k, h, y, ws)  # misaligned x
    N.grouped_ffn(cfg, x, off_t, G, 0, w1, w2k, h, y, ws)  # no rows: nothing to do
    assert N.sync_status(ws) == 0
