"""GPU: the FP8 (E4M3) variant of the expert Linears, called through the C ABI, against
the oracle's statement of the same recipe (per-row E4M3 codes with fp32 scales, fp32
accumulation; h stored in fp16 and quantised per row in turn).

- moe_quantize_e4m3: codes and scales bit for bit (every step is one correctly rounded
  fp32 operation on both sides);
- moe_expert_up_e4m3 / moe_expert_down_e4m3: against fp64 products of the oracle's own
  codes of the same inputs (h and y_perm within one fp16 rounding), on every GEMM plan,
  and the plans against each other bit for bit;
- the whole layer in E4M3 mode against the oracle's E4M3 layer, with the bf16 layers'
  output bound.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_04_b300 import build as B
from routing_dispatch_expert_04_b300 import native as N
from routing_dispatch_expert_04_b300.layer import MoELayer
from routing_dispatch_expert_04_b300.workloads import Workload, make_inputs
from parity_helpers import assert_rounded_to, comparable_tokens, layer_output_error, rel_rms_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    B.build()
    N.lib()


def _decode(codes):
    """E4M3 bytes -> values (torch's float8_e4m3fn view only reinterprets the bytes)."""
    return codes.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_quantize_bit_exact(dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    rows, cols = 300, 512
    m = torch.randn(rows, cols, generator=g, device="cuda") * \
        torch.exp(torch.randn(rows, 1, generator=g, device="cuda") * 3)
    m[7] = 0.0                      # zero row
    m[8, 3] = 1e4                   # one large entry: the rest of the row underflows
    m[9, :] = 2.0 ** -20            # tiny row
    m = m.to(dtype)
    codes = torch.zeros((rows, cols), dtype=torch.uint8, device="cuda")
    scales = torch.zeros(rows, dtype=torch.float32, device="cuda")
    N.quantize_e4m3(m, codes, scales)
    torch.cuda.synchronize()
    want_c, want_s = O.quantize_rows_e4m3(m.float().cpu().numpy())
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(_decode(codes), want_c)


def test_quantize_rows_bounded_on_device():
    m = torch.ones(64, 32, dtype=torch.bfloat16, device="cuda")
    codes = torch.full((64, 32), 0x55, dtype=torch.uint8, device="cuda")
    scales = torch.full((64,), -1.0, device="cuda")
    n = torch.tensor([10], dtype=torch.int32, device="cuda")
    N.quantize_e4m3(m, codes, scales, rows_dev=n)
    torch.cuda.synchronize()
    assert (scales[:10] == 1.0 / 448).all() and (scales[10:] == -1.0).all()
    assert (codes[10:] == 0x55).all()


@pytest.fixture(params=[N.GEMM_SINGLE, N.GEMM_PAIR, N.GEMM_SPLIT, N.GEMM_PAIR_T, N.GEMM_MIXED,
                        N.GEMM_AUTO],
                ids=["single", "pair", "split", "pair_t", "mixed", "auto"])
def pairing(request):
    """Run the E4M3 GEMM on the one-CTA kernel, the CTA-pair kernel, the split of the two,
    the transposed pair kernel, the mixed-tile setting (which E4M3 runs as the split) and
    the default choice."""
    N.set_gemm_pairing(request.param)
    yield request.param
    N.set_gemm_pairing(N.GEMM_AUTO)


def _gen(shape, std, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device="cuda") * std).to(dtype)


@pytest.mark.parametrize("gather", [False, True])
def test_expert_up_e4m3(gather, pairing):
    offs = [0, 300, 300, 812, 813, 1100]
    G, rows, d, F, T, K = 5, 1100, 256, 640, 700, 2
    rows_cap = rows + 16
    cfg = N.make_config(T, d, G, K, F, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    w1 = _gen((G, F, d), d ** -0.5, 2)
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    if gather:
        x = _gen((T, d), 1.0, 1)
        g = torch.Generator(device="cuda")
        g.manual_seed(3)
        src = torch.randint(0, T * K, (rows_cap,), generator=g, device="cuda", dtype=torch.int32)
        a_rows = src.cpu().numpy() // K
    else:
        x = _gen((rows_cap, d), 1.0, 1)
        src = None
        a_rows = np.arange(rows_cap)
    xq = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    sx = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
    w1q = torch.empty((G * F, d), dtype=torch.uint8, device="cuda")
    sw1 = torch.empty(G * F, dtype=torch.float32, device="cuda")
    N.quantize_e4m3(x, xq, sx)
    N.quantize_e4m3(w1.reshape(G * F, d), w1q, sw1)
    h = torch.full((rows_cap, F), 7.0, dtype=torch.float16, device="cuda")
    N.expert_up_e4m3(cfg, xq, sx, src, off_t, G, rows_cap, w1q, sw1, h, ws)
    assert N.sync_status(ws) == 0
    # expected: the oracle's own codes of the same inputs
    cx, sxo = O.quantize_rows_e4m3(to_np(x))
    cw, swo = O.quantize_rows_e4m3(to_np(w1).reshape(G * F, d))
    hn = h.float().cpu().numpy()
    for gi in range(G):
        lo, hi = offs[gi], offs[gi + 1]
        if hi == lo:
            continue
        r = a_rows[lo:hi]
        acc = cx[r] @ cw[gi * F:(gi + 1) * F].T
        ref = O.gelu(acc * sxo[r, None].astype(np.float64) * swo[None, gi * F:(gi + 1) * F])
        assert_rounded_to(hn[lo:hi], ref, "f16")
    assert (hn[rows:] == 7.0).all()


def test_expert_down_e4m3(pairing):
    offs = [0, 129, 129, 700]
    G, rows, F, d = 3, 700, 512, 768
    rows_cap = rows + 8
    cfg = N.make_config(rows, d, G, 1, F, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    h = _gen((rows_cap, F), 0.5, 4, torch.float16)
    w2 = _gen((G, d, F), F ** -0.5, 5)
    hq = torch.empty((rows_cap, F), dtype=torch.uint8, device="cuda")
    sh = torch.empty(rows_cap, dtype=torch.float32, device="cuda")
    w2q = torch.empty((G * d, F), dtype=torch.uint8, device="cuda")
    sw2 = torch.empty(G * d, dtype=torch.float32, device="cuda")
    N.quantize_e4m3(h, hq, sh)
    N.quantize_e4m3(w2.reshape(G * d, F), w2q, sw2)
    y = torch.full((rows_cap, d), 7.0, dtype=torch.float16, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    N.expert_down_e4m3(cfg, hq, sh, off_t, G, rows_cap, w2q, sw2, y, ws)
    assert N.sync_status(ws) == 0
    ch, sho = O.quantize_rows_e4m3(h.float().cpu().numpy())
    cw, swo = O.quantize_rows_e4m3(to_np(w2).reshape(G * d, F))
    yn = y.float().cpu().numpy()
    for gi in range(G):
        lo, hi = offs[gi], offs[gi + 1]
        if hi == lo:
            continue
        ref = (ch[lo:hi] @ cw[gi * d:(gi + 1) * d].T) * sho[lo:hi, None].astype(np.float64) \
            * swo[None, gi * d:(gi + 1) * d]
        assert_rounded_to(yn[lo:hi], ref, "f16")
    assert (yn[rows:] == 7.0).all()


@pytest.mark.parametrize("fn", ["up", "down"])
def test_e4m3_plans_agree_bitwise(fn):
    """The one-CTA kernel, the CTA-pair kernel, their split and the transposed pairs
    multiply the same E4M3 codes and accumulate the 128-deep k-blocks in the same order:
    outputs bit for bit."""
    offs = [0, 300, 812, 813, 1400]
    G, rows, Kd, Nn = 4, 1400, 512, 768
    rows_cap = rows + 16
    cfg = N.make_config(rows, Kd if fn == "up" else Nn, G, 1, Nn if fn == "up" else Kd, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    a = _gen((rows_cap, Kd), 1.0, 21, torch.bfloat16 if fn == "up" else torch.float16)
    w = _gen((G * Nn, Kd), Kd ** -0.5, 22)
    aq = torch.empty((rows_cap, Kd), dtype=torch.uint8, device="cuda")
    sa = torch.empty(rows_cap, dtype=torch.float32, device="cuda")
    wq = torch.empty((G * Nn, Kd), dtype=torch.uint8, device="cuda")
    sw = torch.empty(G * Nn, dtype=torch.float32, device="cuda")
    N.quantize_e4m3(a, aq, sa)
    N.quantize_e4m3(w, wq, sw)
    outs = []
    for mode in (N.GEMM_SINGLE, N.GEMM_PAIR, N.GEMM_SPLIT, N.GEMM_PAIR_T):
        N.set_gemm_pairing(mode)
        try:
            out = torch.zeros((rows_cap, Nn), dtype=torch.float16, device="cuda")
            if fn == "up":
                N.expert_up_e4m3(cfg, aq, sa, None, off_t, G, rows_cap, wq, sw, out, ws)
            else:
                N.expert_down_e4m3(cfg, aq, sa, off_t, G, rows_cap, wq, sw, out, ws)
        finally:
            N.set_gemm_pairing(N.GEMM_AUTO)
        assert N.sync_status(ws) == 0
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], outs[2])
    assert torch.equal(outs[0], outs[3])


FP8_LAYERS = [
    Workload("fp8_small", 300, 256, 8, 2, 384, "bf16", 1.25),
    Workload("fp8_bias_shared", 333, 128, 32, 8, 96, "bf16", None, bias="normal", shared=True),
    Workload("fp8_zipf", 1000, 192, 8, 2, 256, "bf16", 1.0, bias="zipf"),
]


@pytest.mark.parametrize("fused", [False, True], ids=["copy_dispatch", "fused_dispatch"])
@pytest.mark.parametrize("wl", FP8_LAYERS, ids=[w.name for w in FP8_LAYERS])
def test_layer_e4m3(wl, fused):
    """Whole layer with E4M3 experts, fed the oracle's logits: routing bit for bit and
    the output within the bf16 layers' bound of the oracle's E4M3 layer.  The distance to
    the exact (non-FP8) layer is printed: it is the FP8 rounding itself."""
    inp = make_inputs(wl, "cuda")
    layer = MoELayer.from_workload(wl, inp, experts="e4m3", fused_dispatch=fused)
    x_np = to_np(inp["x"])
    b_np = None if inp["b_r"] is None else to_np(inp["b_r"])
    _, L32 = O.router_logits(x_np, to_np(inp["w_r"]), b_np)
    layer.forward(inp["x"], logits_in=torch.from_numpy(L32).cuda())
    layer.check_device_status()
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    shared = (to_np(inp["w1s"])[0], to_np(inp["w2s"])[0]) if wl.shared else None
    args = (x_np, to_np(inp["w_r"]), b_np, to_np(inp["w1"]), to_np(inp["w2"]), wl.K, C, wl.alpha)
    ref8 = O.moe_forward(*args, shared=shared, logits32=L32, experts="e4m3")
    ref = O.moe_forward(*args, shared=shared, logits32=L32)
    assert np.array_equal(to_np(layer.ids), ref8["ids"])
    assert np.array_equal(to_np(layer.slot), ref8["slot"].reshape(wl.T, wl.K))
    y = to_np(layer.y)
    err, literal = layer_output_error(y, ref8["y"], "bf16")
    rms_vs_exact = float(np.sqrt(np.mean((y - ref["y"]) ** 2)) / np.sqrt(np.mean(ref["y"] ** 2)))
    print(f"{wl.name}: vs E4M3 oracle {err:.4g} (literal {literal:.4g}); "
          f"RMS distance to the exact layer {rms_vs_exact:.4g}")
    assert err <= 2e-2, (err, literal)
