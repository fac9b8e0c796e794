"""GPU parity of the routed-expert layer (W4A16 and W4A4) and the dense
linear against the oracle.  Tolerance: relative L2 error <= 5e-3 and every
element within 2e-2 * rms(oracle out), or the bf16 neighbour of the
oracle's value where its unrounded value lies within the derived error
bound of the midpoint (tests/gpu_util.py); the kernels' h is checked on the
way (tests/layer_check.py).  Every test that picks a kernel asserts, from
the library's launch names, that the kernel it meant ran."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from gpu_util import OracleBank, assert_bank_equal, bf16_to_f32, gpu_bank, kernels_ran, pick_tokens
from layer_check import check_layer, check_linear_h, check_linear_y
from oracle import calib
from serving_nvfp4_routed_gb300 import synth

pytestmark = pytest.mark.gpu

FULL = synth.MoEShape(T=64, d=4096, E=288, k=8, F=1536)


def tc_possible(mode, d, F):
    if mode == "w4a16":
        return d % 128 == 0 and F % 128 == 0
    return d % 256 == 0 and F % 256 == 0  # the block-scaled FP4 kernels: K a multiple of 256


def expected_family(path, mode, T, E, k, d, F):
    if not tc_possible(mode, d, F) or path.startswith("gemv"):
        return "gemv"
    if path == "tc":
        return "tc"
    R = T * k
    return "tc" if R >= 32 * min(E, R) else "gemv"


def bf16_rows(fam, mode, d, F):
    """Whether the path keeps each routed row's y in bf16 for the ordered
    combine (the R3 rounding point): every prompt-shaped (tensor-core)
    path does."""
    return fam == "tc"


def assert_decode_form(names, path, d, F, what=""):
    """A forced decode-shaped form ran: one persistent launch where d and F
    are multiples of 256, else (and when the two launches are forced) the
    gate/up and down GEMV launches."""
    fused = [n for n in names if "gateup_down" in n]
    if path == "gemv_split" or (path == "gemv_fused" and (d % 256 or F % 256)):
        assert not fused, f"{what}: expected the two-launch form, launched {sorted(names)}"
    elif path == "gemv_fused":
        assert fused, f"{what}: expected the one-launch form, launched {sorted(names)}"


def assert_family(names, fam, what=""):
    pre = ("gemv_",) if fam == "gemv" else ("tc_", "tcm_", "tcq_")
    gate = [n for n in names if n.startswith(pre) and "gateup" in n]
    down = [n for n in names if n.startswith(pre) and "down" in n]
    assert gate and down, f"{what}: expected {fam} gate/up and down kernels, launched {sorted(names)}"
    other = ("tc_", "tcm_", "tcq_") if fam == "gemv" else ("gemv_",)
    assert not [n for n in names if n.startswith(other)], f"{what}: unexpected kernels {sorted(names)}"


@pytest.fixture(params=["auto", "gemv_split", "gemv_fused", "tc"])
def path(request):
    """Run the test with the library's own choice of kernel and with each
    kernel forced (the tensor-core path needs d and F multiples of 128;
    W4A4 on the tensor cores multiples of 256; the one-launch decode form
    d and F multiples of 256)."""
    lib.set_kernel_choice(request.param)
    yield request.param
    lib.set_kernel_choice("auto")


def _small(orc, shape, seed, outlier=0.0, kind="normal"):
    inp = synth.moe_inputs(shape, seed, device="cuda", outlier_frac=outlier, logits_kind=kind)
    banks = dict(gate=inp["gate"], up=inp["up"], down=inp["down"])
    gw = gpu_bank(lib, banks)
    ob = OracleBank(orc, banks).get()
    assert_bank_equal(gw, ob, range(shape.E))
    return inp, gw, ob


def _run(mode, x, logits, k, gw, is13=None, is2=None, ws=None):
    T, d = x.shape
    if ws is None:
        ws = lib.moe_workspace(T, gw.E, k, d, gw.F, mode, "cuda")
    if mode == "w4a16":
        fn = lambda: lib.nvfp4_moe_w4a16(x, logits, k, gw, ws=ws)
    else:
        fn = lambda: lib.nvfp4_moe_w4a4(x, logits, k, gw, torch.from_numpy(is13).cuda(),
                                        torch.from_numpy(is2).cuda(), ws=ws)
    out, names = kernels_ran(lib, fn)
    return out, ws, names


def _calibrate(orc, shape, ob, seed, **kw):
    """Static input scales from a seeded calibration draw of the layer's own
    input distribution (p99 of the routed rows' block maxima x 1.05 / 2688
    per expert and projection, the oracle computing h): 1024 tokens for the
    full-size layer, 64 for the tiny one."""
    n = 1024 if shape.E > 64 else 64
    x = synth.make_x(n, shape.d, seed, outlier_frac=0.05)
    lg = synth.make_logits(n, shape.E, seed + 1)
    return calib.calibrate(synth.bf16_bits(x), lg.numpy(), shape.k, ob, **kw)


@pytest.mark.parametrize("mode", ["w4a16", "w4a4"])
def test_tiny(orc, path, mode):
    s = synth.TINY
    inp, gw, ob = _small(orc, s, seed=1000)
    is13 = is2 = None
    if mode == "w4a4":
        is13, is2 = _calibrate(orc, s, ob, 1999)
    out, ws, names = _run(mode, inp["x"], inp["logits"], s.k, gw, is13, is2)
    fam = expected_family(path, mode, s.T, s.E, s.k, s.d, s.F)
    assert_family(names, fam, f"tiny {mode} {path}")
    assert_decode_form(names, path, s.d, s.F, f"tiny {mode} {path}")
    check_layer(orc, mode, inp["x"], inp["logits"], s.k, ob, out, ws, np.arange(s.T, dtype=np.int32), is13, is2,
                f"tiny {mode} {path}", round_y=bf16_rows(fam, mode, s.d, s.F))


@pytest.mark.parametrize("T,E,k,d,F", [(13, 8, 2, 256, 128), (40, 16, 4, 512, 256), (3, 5, 5, 192, 64),
                                       (100, 32, 8, 1024, 320), (300, 6, 2, 512, 256)])
def test_ragged_shapes_both_modes(orc, T, E, k, d, F, path):
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob = _small(orc, s, seed=T + E, outlier=0.05)
    tok = np.arange(T, dtype=np.int32)
    xb = synth.bf16_bits(inp["x"])
    out, ws, names = _run("w4a16", inp["x"], inp["logits"], k, gw)
    fam = expected_family(path, "w4a16", T, E, k, d, F)
    assert_family(names, fam, "w4a16")
    assert_decode_form(names, path, d, F, "w4a16")
    check_layer(orc, "w4a16", inp["x"], inp["logits"], k, ob, out, ws, tok, what=f"w4a16 {path}",
                round_y=bf16_rows(fam, "w4a16", d, F))
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob)
    out4, ws4, names4 = _run("w4a4", inp["x"], inp["logits"], k, gw, is13, is2)
    fam4 = expected_family(path, "w4a4", T, E, k, d, F)
    assert_family(names4, fam4, "w4a4")
    assert_decode_form(names4, path, d, F, "w4a4")
    check_layer(orc, "w4a4", inp["x"], inp["logits"], k, ob, out4, ws4, tok, is13, is2, f"w4a4 {path}",
                round_y=bf16_rows(fam4, "w4a4", d, F))


# ---------------------------------------------------------------------------
# full-size layer: E=288, top-8, d=4096, ffn=1536
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def full(orc):
    s = FULL
    banks = dict(gate=synth.make_weights(s.E, s.F, s.d, 1013, "cuda"),
                 up=synth.make_weights(s.E, s.F, s.d, 1014, "cuda"),
                 down=synth.make_weights(s.E, s.d, s.F, 1015, "cuda"))
    gw = gpu_bank(lib, banks)
    return banks, gw, OracleBank(orc, banks)


@pytest.fixture(scope="module")
def full_calibration(orc, full):
    """The W4A4 static scales of the full-size layer: per expert and
    projection, p99 of the block maxima of the rows routed to it in a seeded
    1024-token draw (5 % outlier rows, as the prompt workloads), x 1.05 /
    2688 (W4A4 model card, "Quantization boundary")."""
    banks, gw, bank = full
    ob = bank.get()  # every expert: the draw reaches all of them
    return _calibrate(orc, FULL, ob, 7001)


def _full_case(orc, full, mode, T, kind, outlier, seed, scales=None, n_tok=32, fam="tc", form=None):
    banks, gw, bank = full
    s = FULL
    x = synth.make_x(T, s.d, seed, "cuda", outlier_frac=outlier)
    logits = synth.make_logits(T, s.E, seed + 1, "cuda", kind=kind)
    r = orc.route(logits.cpu().numpy(), s.k)
    tok = np.arange(T, dtype=np.int32) if T <= n_tok else pick_tokens(r, T, s.k, n=n_tok, seed=seed)
    experts = np.unique(r["ids"][tok])
    ob = bank.get(experts)
    assert_bank_equal(gw, ob, experts)
    is13, is2 = scales if scales is not None else (None, None)
    out, ws, names = _run(mode, x, logits, s.k, gw, is13, is2)
    assert_family(names, fam, f"{mode} T={T} {kind}")
    if form:
        assert_decode_form(names, form, s.d, s.F, f"{mode} T={T} {kind}")
    return check_layer(orc, mode, x, logits, s.k, ob, out, ws, tok, is13, is2, f"{mode} T={T} {kind}",
                       round_y=bf16_rows(fam, mode, s.d, s.F))


@pytest.fixture(params=["gemv_split", "gemv_fused"])
def decode_form(request):
    lib.set_kernel_choice(request.param)
    yield request.param
    lib.set_kernel_choice("auto")


@pytest.mark.parametrize("T", (1, 2) + tuple(synth.DECODE_T[1:]))
def test_decode_w4a16_every_token(orc, full, T, decode_form):
    """Decode-shaped layer at full size, in each of its two forms; every
    token against the oracle (T=2: the gate/up items of 32 features with K
    over four warp quarters)."""
    _full_case(orc, full, "w4a16", T, "normal", 0.0, 1011 + T, n_tok=64, fam="gemv", form=decode_form)


@pytest.mark.parametrize("T", [8, 32])
def test_decode_w4a4_calibrated(orc, full, full_calibration, T, decode_form):
    _full_case(orc, full, "w4a4", T, "normal", 0.05, 2001 + T, full_calibration, n_tok=64, fam="gemv",
               form=decode_form)


@pytest.mark.parametrize("mode", ["w4a16", "w4a4"])
def test_decode_deterministic(full, decode_form, mode):
    """The decode-shaped combine sums each token's rows in slot order: two
    calls on the same inputs give the same bits."""
    banks, gw, bank = full
    s = FULL
    x = synth.make_x(64, s.d, 3301, "cuda")
    lg = synth.make_logits(64, s.E, 3302, "cuda")
    if mode == "w4a16":
        run = lambda: lib.nvfp4_moe_w4a16(x, lg, s.k, gw)
    else:
        sc = torch.full((s.E,), 0.01, dtype=torch.float32, device="cuda")
        run = lambda: lib.nvfp4_moe_w4a4(x, lg, s.k, gw, sc, sc)
    a = run()
    b = run()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T", [1, 64])
def test_decode_shapes_on_tensor_cores(orc, full, T):
    """The prompt-shaped kernels (forced) at decode batch sizes."""
    lib.set_kernel_choice("tc")
    try:
        _full_case(orc, full, "w4a16", T, "normal", 0.0, 2101 + T, n_tok=64, fam="tc")
    finally:
        lib.set_kernel_choice("auto")


@pytest.mark.parametrize("mode,T,kind", [("w4a16", 4096, "normal"), ("w4a4", 8192, "normal"),
                                         ("w4a16", 16384, "zipf"), ("w4a4", 16384, "zipf"),
                                         ("w4a16", 16384, "zipf_masked"), ("w4a4", 16384, "zipf_masked")])
def test_prefill_full_size(orc, full, full_calibration, mode, T, kind):
    """Prompt-shaped layers at full size: W4A16 at T=4096 and W4A4 at
    T=8192 with 5 % outlier rows x 8, skewed Zipf(1.2) popularity at
    T=16384 (and a third of the experts masked off); W4A4 with the
    calibrated static scales.  At least 32 tokens against the oracle,
    covering the first and last row tile of the most popular expert and the
    rows of the least popular one."""
    outlier = 0.05 if kind == "normal" else 0.0
    rep = _full_case(orc, full, mode, T, kind, outlier, 3001 + T + len(kind),
                     full_calibration if mode == "w4a4" else None)
    assert rep["n"] >= 32 * 4096


def test_given_routing_and_bad_ids(orc):
    """logits=None uses the routing arrays in the workspace; an out-of-range
    id is reported through d_status and does not fault."""
    s = synth.TINY
    inp, gw, ob = _small(orc, s, seed=1000)
    r = orc.route(inp["logits"].cpu().numpy(), s.k)
    ws = lib.moe_workspace(s.T, s.E, s.k, s.d, s.F, "w4a16", "cuda")
    v = lib.moe_workspace_views(ws, s.T, s.E, s.k, s.d, s.F, "w4a16")
    v["ids"].copy_(torch.from_numpy(r["ids"]))
    v["w"].copy_(torch.from_numpy(r["w"]))
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = lib.nvfp4_moe_w4a16(inp["x"], None, s.k, gw, ws=ws, d_status=st)
    check_layer(orc, "w4a16", inp["x"], inp["logits"], s.k, ob, out, ws, np.arange(s.T, dtype=np.int32),
                what="given routing")
    assert st[0].item() == 0
    assert np.array_equal(v["row_to_slot"].cpu().numpy(), r["row_to_slot"])
    v["ids"].copy_(torch.from_numpy(r["ids"]))
    v["ids"][1, 0] = s.E + 5
    lib.nvfp4_moe_w4a16(inp["x"], None, s.k, gw, ws=ws, d_status=st)
    torch.cuda.synchronize()
    assert st[0].item() == 8  # NVFP4_ERR_DEVICE_INPUT


def test_zero_tokens():
    s = synth.TINY
    gw = gpu_bank(lib, dict(gate=synth.make_weights(s.E, s.F, s.d, 1, "cuda"),
                            up=synth.make_weights(s.E, s.F, s.d, 2, "cuda"),
                            down=synth.make_weights(s.E, s.d, s.F, 3, "cuda")))
    out = lib.nvfp4_moe_w4a16(torch.zeros(0, s.d, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(0, s.E, device="cuda"), s.k, gw)
    assert out.shape == (0, s.d)


def _dense(orc, M, K, N, seed, rows=None, up_scale=3.0, fam=None):
    x = synth.make_x(M, K, seed=seed, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, N, K, seed + 1, "cuda")[0]
    wu = synth.make_weights(1, N, K, seed + 2, "cuda")[0] * up_scale  # different tensor scale
    wd = synth.make_weights(1, K, N, seed + 3, "cuda")[0]
    qg, qu, qd = (lib.nvfp4_quantize_weights(w) for w in (wg, wu, wd))
    og, ou, od = (orc.quantize_tensor(synth.bf16_bits(w)) for w in (wg, wu, wd))
    for q, o in ((qg, og), (qu, ou), (qd, od)):
        assert np.array_equal(q.codes[0].cpu().numpy(), o[0]) and q.weight_scale_2.item() == o[2]
    assert qg.weight_scale_2.item() != qu.weight_scale_2.item()
    rows = np.arange(M) if rows is None else rows
    h, names = kernels_ran(lib, lambda: lib.nvfp4_linear(x, qg, qu))
    if fam:
        pre = ("gemv_",) if fam == "gemv" else ("tc_", "tcm_")
        assert any(n.startswith(pre) for n in names), (fam, names)
    ex, _ = check_linear_h(orc, x[torch.from_numpy(rows).cuda()], og, ou, bf16_to_f32(h)[rows], "dense gate/up")
    # down projection on the oracle's own h, so that only its own sums differ
    href = torch.from_numpy(ex["out"]).to(torch.bfloat16)
    hin = torch.zeros(M, N, dtype=torch.bfloat16)
    hin[torch.from_numpy(rows)] = href
    y = lib.nvfp4_linear(hin.cuda(), qd)
    check_linear_y(orc, synth.bf16_bits(href), od, bf16_to_f32(y)[rows], "dense down")


@pytest.mark.parametrize("M,K,N", [(7, 256, 128), (64, 1024, 512), (130, 512, 192), (300, 256, 384)])
def test_dense_linear_and_mlp(orc, M, K, N, path):
    fam = None if path == "auto" else ("gemv" if path.startswith("gemv") or N % 128 else "tc")
    _dense(orc, M, K, N, M, fam=fam)


def test_dense_mlp_full_size_sampled(orc):
    """Dense NVFP4 MLP d=4096, ffn=12288, 8192 tokens; gate and up carry
    different tensor scales; 40 rows from many 128-row tiles (and the first
    and last) against the oracle."""
    M = synth.DENSE["M"]
    rows = np.unique(np.append(np.random.default_rng(4005).choice(M, 38, replace=False), [0, M - 1]))
    _dense(orc, M, synth.DENSE["d"], synth.DENSE["F"], 4001, rows=rows, up_scale=2.0, fam="tc")


def test_linear_many_units_per_cta(orc):
    """Single-projection linear with 8192 rows, K=1536, N=4096: every CTA of
    the prompt-shaped kernel works through several (row tile, column slice)
    units, so ring slots are refilled many times; 40 rows against the
    oracle."""
    M, K, N = 8192, 1536, 4096
    x = synth.make_x(M, K, seed=4101, device="cuda", outlier_frac=0.05)
    w = synth.make_weights(1, N, K, 4102, "cuda")[0]
    q = lib.nvfp4_quantize_weights(w)
    y, names = kernels_ran(lib, lambda: lib.nvfp4_linear(x, q))
    assert any(n.startswith("tcm_linear") for n in names), names
    rows = np.unique(np.append(np.random.default_rng(4103).choice(M, 38, replace=False), [0, M - 1]))
    oq = orc.quantize_tensor(synth.bf16_bits(w))
    check_linear_y(orc, synth.bf16_bits(x)[rows], oq, bf16_to_f32(y)[rows], "linear K=1536 N=4096")


@pytest.mark.parametrize("T,E,k,d,F", [(512, 16, 4, 512, 256), (300, 6, 2, 1024, 512)])
def test_prompt_w4a4_tensor_cores(orc, T, E, k, d, F):
    """W4A4 through the prompt-shaped block-scaled FP4 kernels (forced),
    several work units per expert (and a last 192-wide column slice that
    reaches past d), against the oracle on every token."""
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob = _small(orc, s, seed=T + 7, outlier=0.05)
    xb = synth.bf16_bits(inp["x"])
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob)
    lib.set_kernel_choice("tc")
    try:
        out, ws, names = _run("w4a4", inp["x"], inp["logits"], k, gw, is13, is2)
    finally:
        lib.set_kernel_choice("auto")
    assert any(n.startswith("tcq_gateup") for n in names) and any(n.startswith("tcq_down") for n in names), names
    check_layer(orc, "w4a4", inp["x"], inp["logits"], k, ob, out, ws, np.arange(T, dtype=np.int32), is13, is2,
                "prompt w4a4", round_y=True)


@pytest.mark.parametrize("mode,F", [("w4a16", 256), ("w4a4", 256), ("w4a16", 384)])
def test_prompt_deterministic_and_chunk_invariant(orc, mode, F):
    """The prompt-shaped path (forced) gives the same bits on every call and
    for any chunking of the batch: each routed row's result depends only on
    its own data (fixed K order, per-row scale), and each token's k weighted
    rows are summed in slot order.  ffn 384 takes the weights-as-M kernel
    for the down projection (K not a multiple of 256)."""
    T, E, k, d = 512, 16, 4, 512
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob = _small(orc, s, seed=T + 23, outlier=0.05)
    x, lg = inp["x"], inp["logits"]
    if mode == "w4a16":
        run = lambda xx, ll: lib.nvfp4_moe_w4a16(xx, ll, k, gw)
    else:
        xb = synth.bf16_bits(x)
        is13, is2 = calib.calibrate(xb, lg.cpu().numpy(), k, ob)
        is13, is2 = torch.from_numpy(is13).cuda(), torch.from_numpy(is2).cuda()
        run = lambda xx, ll: lib.nvfp4_moe_w4a4(xx, ll, k, gw, is13, is2)
    lib.set_kernel_choice("tc")
    try:
        full = run(x, lg)
        again = run(x, lg)
        parts = torch.cat([run(x[:200].contiguous(), lg[:200].contiguous()),
                           run(x[200:].contiguous(), lg[200:].contiguous())])
    finally:
        lib.set_kernel_choice("auto")
    assert torch.equal(full.view(torch.int16), again.view(torch.int16))
    assert torch.equal(full.view(torch.int16), parts.view(torch.int16))


@pytest.mark.parametrize("layer", [5, 30])
@pytest.mark.parametrize("kpath", ["gemv", "tc"])
def test_w4a4_layer_specific_calibration(orc, layer, kpath):
    """W4A4 with the card's layer-specific w2 percentiles (p98 at layer 5,
    p98.9 at layer 30) on the decode and the prompt kernels, every token
    against the oracle."""
    T, E, k, d, F = 256, 16, 4, 512, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob = _small(orc, s, seed=layer + 61, outlier=0.05)
    xb = synth.bf16_bits(inp["x"])
    p13, p2 = calib.layer_percentiles(layer)
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob, pct13=p13, pct2=p2)
    lib.set_kernel_choice(kpath)
    try:
        out, ws, names = _run("w4a4", inp["x"], inp["logits"], k, gw, is13, is2)
    finally:
        lib.set_kernel_choice("auto")
    assert_family(names, kpath, f"layer {layer} {kpath}")
    check_layer(orc, "w4a4", inp["x"], inp["logits"], k, ob, out, ws, np.arange(T, dtype=np.int32), is13, is2,
                f"w4a4 layer {layer} {kpath}", round_y=bf16_rows(kpath, "w4a4", d, F))
