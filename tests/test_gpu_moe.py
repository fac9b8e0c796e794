"""GPU parity of the routed-expert layer (W4A16 and W4A4) and the dense
linear against the oracle, with the tolerance the layer is held to:
relative L2 error <= 5e-3 and max abs error <= 2e-2 * rms(oracle out)."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from oracle import calib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import assert_bank_equal, assert_layer_close, bf16_to_f32, gpu_bank, oracle_bank

pytestmark = pytest.mark.gpu


def _setup(orc, shape, seed, outlier=0.0, kind="normal", experts_for=None):
    inp = synth.moe_inputs(shape, seed, device="cuda", outlier_frac=outlier, logits_kind=kind)
    banks = dict(gate=inp["gate"], up=inp["up"], down=inp["down"])
    gw = gpu_bank(lib, banks)
    r = orc.route(inp["logits"].cpu().numpy(), shape.k)
    tokens = experts_for if experts_for is not None else np.arange(shape.T)
    experts = np.arange(shape.E) if shape.E <= 64 else np.unique(r["ids"][tokens])
    ob = oracle_bank(orc, banks, experts)
    assert_bank_equal(gw, ob, experts)
    return inp, gw, ob, r, np.asarray(tokens, np.int32)


@pytest.fixture(params=["auto", "gemv", "tc"])
def path(request, monkeypatch):
    """Run the test with the library's own choice of kernel and with each
    kernel forced (the tensor-core path needs d and F multiples of 128)."""
    if request.param == "auto":
        monkeypatch.delenv("NVFP4_PATH", raising=False)
    else:
        monkeypatch.setenv("NVFP4_PATH", request.param)
    return request.param


def test_tiny_w4a16(orc, path):
    s = synth.TINY
    inp, gw, ob, r, tok = _setup(orc, s, seed=1000)
    out = lib.nvfp4_moe_w4a16(inp["x"], inp["logits"], s.k, gw)
    ref = orc.moe_layer("w4a16", synth.bf16_bits(inp["x"]), r["ids"], r["w"], ob)
    assert_layer_close(bf16_to_f32(out), ref, "tiny w4a16")


def test_tiny_w4a4(orc):
    s = synth.TINY
    inp, gw, ob, r, tok = _setup(orc, s, seed=1000)
    cal = synth.moe_inputs(synth.MoEShape(64, s.d, s.E, s.k, s.F), 1999)
    is13, is2 = calib.calibrate(synth.bf16_bits(cal["x"]), cal["logits"].numpy(), s.k, ob)
    out = lib.nvfp4_moe_w4a4(inp["x"], inp["logits"], s.k, gw, torch.from_numpy(is13).cuda(),
                             torch.from_numpy(is2).cuda())
    ref = orc.moe_layer("w4a4", synth.bf16_bits(inp["x"]), r["ids"], r["w"], ob, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out), ref, "tiny w4a4")


@pytest.mark.parametrize("T,E,k,d,F", [(13, 8, 2, 256, 128), (40, 16, 4, 512, 256), (3, 5, 5, 192, 64),
                                       (100, 32, 8, 1024, 320)])
def test_ragged_shapes_both_modes(orc, T, E, k, d, F, path):
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob, r, tok = _setup(orc, s, seed=T + E, outlier=0.05)
    xb = synth.bf16_bits(inp["x"])
    out = lib.nvfp4_moe_w4a16(inp["x"], inp["logits"], k, gw)
    ref = orc.moe_layer("w4a16", xb, r["ids"], r["w"], ob)
    assert_layer_close(bf16_to_f32(out), ref, "w4a16")
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob)
    out4 = lib.nvfp4_moe_w4a4(inp["x"], inp["logits"], k, gw, torch.from_numpy(is13).cuda(),
                              torch.from_numpy(is2).cuda())
    ref4 = orc.moe_layer("w4a4", xb, r["ids"], r["w"], ob, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out4), ref4, "w4a4")


@pytest.fixture(scope="module")
def decode_bank():
    s = synth.decode(64)
    banks = dict(gate=synth.make_weights(s.E, s.F, s.d, 1013, "cuda"),
                 up=synth.make_weights(s.E, s.F, s.d, 1014, "cuda"),
                 down=synth.make_weights(s.E, s.d, s.F, 1015, "cuda"))
    gw = gpu_bank(lib, banks)
    return banks, gw


@pytest.mark.parametrize("T", synth.DECODE_T)
def test_decode_w4a16_sampled(orc, decode_bank, T):
    """Decode-shaped layer at full size; oracle on a seeded sample of tokens."""
    banks, gw = decode_bank
    s = synth.decode(T)
    x = synth.make_x(T, s.d, 1011 + T, "cuda")
    logits = synth.make_logits(T, s.E, 1012 + T, "cuda")
    out = lib.nvfp4_moe_w4a16(x, logits, s.k, gw)
    r = orc.route(logits.cpu().numpy(), s.k)
    rng = np.random.default_rng(T)
    tok = np.sort(rng.choice(T, size=min(T, 3), replace=False)).astype(np.int32)
    experts = np.unique(r["ids"][tok])
    ob = oracle_bank(orc, banks, experts)
    assert_bank_equal(gw, ob, experts)
    ref = orc.moe_layer("w4a16", synth.bf16_bits(x), r["ids"], r["w"], ob, tokens=tok)
    assert_layer_close(bf16_to_f32(out)[tok], ref, f"decode T={T}")


def test_decode_w4a4_sampled(orc, decode_bank):
    banks, gw = decode_bank
    s = synth.decode(32)
    x = synth.make_x(s.T, s.d, 2001, "cuda", outlier_frac=0.05)
    logits = synth.make_logits(s.T, s.E, 2002, "cuda")
    r = orc.route(logits.cpu().numpy(), s.k)
    tok = np.array([0, 17], np.int32)
    experts = np.unique(r["ids"][tok])
    ob = oracle_bank(orc, banks, experts)
    rng = np.random.default_rng(5)
    is13 = (rng.uniform(0.5, 1.5, s.E) * 4.0 / 2688).astype(np.float32)
    is2 = (rng.uniform(0.5, 1.5, s.E) * 1.0 / 2688).astype(np.float32)
    out = lib.nvfp4_moe_w4a4(x, logits, s.k, gw, torch.from_numpy(is13).cuda(), torch.from_numpy(is2).cuda())
    ref = orc.moe_layer("w4a4", synth.bf16_bits(x), r["ids"], r["w"], ob, tokens=tok, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out)[tok], ref, "decode w4a4")


def test_given_routing_and_bad_ids(orc):
    """logits=None uses the routing arrays in the workspace; an out-of-range
    id is reported through d_status and does not fault."""
    s = synth.TINY
    inp, gw, ob, r, tok = _setup(orc, s, seed=1000)
    ws = lib.moe_workspace(s.T, s.E, s.k, s.d, s.F, "w4a16", "cuda")
    v = lib.moe_workspace_views(ws, s.T, s.E, s.k, s.d, s.F, "w4a16")
    v["ids"].copy_(torch.from_numpy(r["ids"]))
    v["w"].copy_(torch.from_numpy(r["w"]))
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = lib.nvfp4_moe_w4a16(inp["x"], None, s.k, gw, ws=ws, d_status=st)
    ref = orc.moe_layer("w4a16", synth.bf16_bits(inp["x"]), r["ids"], r["w"], ob)
    assert_layer_close(bf16_to_f32(out), ref, "given routing")
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


@pytest.mark.parametrize("M,K,N", [(7, 256, 128), (64, 1024, 512), (130, 512, 192), (300, 256, 384)])
def test_dense_linear_and_mlp(orc, M, K, N, path):
    x = synth.make_x(M, K, seed=M, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, N, K, 10 + M, "cuda")[0]
    wu = synth.make_weights(1, N, K, 20 + M, "cuda")[0] * 3  # different tensor scale
    wd = synth.make_weights(1, K, N, 30 + M, "cuda")[0]
    qg, qu, qd = (lib.nvfp4_quantize_weights(w) for w in (wg, wu, wd))
    og, ou, od = (orc.quantize_tensor(synth.bf16_bits(w)) for w in (wg, wu, wd))
    assert qg.weight_scale_2.item() != qu.weight_scale_2.item()
    h = lib.nvfp4_linear(x, qg, qu)
    href = orc.linear(synth.bf16_bits(x), og[0], og[1], og[2], wup=ou)
    assert_layer_close(bf16_to_f32(h), href, "gate/up")
    y = lib.nvfp4_linear(h, qd)
    href_bits = synth.bf16_bits(torch.from_numpy(href).to(torch.bfloat16))  # the oracle's own h
    yref = orc.linear(href_bits, od[0], od[1], od[2])
    assert_layer_close(bf16_to_f32(y), yref, "down")


@pytest.mark.parametrize("kind,mode", [("normal", "w4a16"), ("zipf", "w4a16"), ("zipf_masked", "w4a16"),
                                       ("normal", "w4a4"), ("zipf", "w4a4")])
def test_prefill_sampled(orc, decode_bank, kind, mode):
    """Prompt-shaped layers at full size (T=4096 for W4A16, skewed popularity
    at T=16384, W4A4 at T=8192 with 5 % outlier rows); the oracle evaluates
    a seeded sample of tokens."""
    banks, gw = decode_bank
    T = {"normal": 4096 if mode == "w4a16" else 8192, "zipf": 16384, "zipf_masked": 16384}[kind]
    s = synth.MoEShape(T, 4096, 288, 8, 1536)
    x = synth.make_x(T, s.d, 3001 + T, "cuda", outlier_frac=0.05)
    logits = synth.make_logits(T, s.E, 3002 + T, "cuda", kind=kind)
    r = orc.route(logits.cpu().numpy(), s.k)
    rng = np.random.default_rng(T)
    tok = np.sort(rng.choice(T, size=2, replace=False)).astype(np.int32)
    if kind != "normal":
        # include the most popular expert's first token
        top = np.argmax(np.diff(r["offsets"]))
        tok = np.unique(np.append(tok, np.where((r["ids"] == top).any(1))[0][0])).astype(np.int32)
    experts = np.unique(r["ids"][tok])
    ob = oracle_bank(orc, banks, experts)
    if mode == "w4a16":
        out = lib.nvfp4_moe_w4a16(x, logits, s.k, gw)
        ref = orc.moe_layer("w4a16", synth.bf16_bits(x), r["ids"], r["w"], ob, tokens=tok)
    else:
        rs = np.random.default_rng(6)
        is13 = (rs.uniform(0.5, 1.5, s.E) * 20.0 / 2688).astype(np.float32)
        is2 = (rs.uniform(0.5, 1.5, s.E) * 4.0 / 2688).astype(np.float32)
        out = lib.nvfp4_moe_w4a4(x, logits, s.k, gw, torch.from_numpy(is13).cuda(), torch.from_numpy(is2).cuda())
        ref = orc.moe_layer("w4a4", synth.bf16_bits(x), r["ids"], r["w"], ob, tokens=tok, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out)[tok], ref, f"prefill {kind} {mode}")


def test_dense_mlp_full_size_sampled(orc):
    """Dense NVFP4 MLP d=4096, ffn=12288, 8192 tokens; gate and up carry
    different tensor scales; the oracle checks sampled rows."""
    M, K, N = 8192, 4096, 12288
    x = synth.make_x(M, K, seed=4001, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, N, K, 4002, "cuda")[0]
    wu = synth.make_weights(1, N, K, 4003, "cuda")[0] * 2
    wd = synth.make_weights(1, K, N, 4004, "cuda")[0]
    qg, qu, qd = (lib.nvfp4_quantize_weights(w) for w in (wg, wu, wd))
    h = lib.nvfp4_linear(x, qg, qu)
    y = lib.nvfp4_linear(h, qd)
    # rows from many 128-row tiles: a CTA's later work units get checked too
    rows = np.unique(np.append(np.random.default_rng(4005).choice(M, 22, replace=False), [0, M - 1]))
    og, ou, od = (orc.quantize_tensor(synth.bf16_bits(w)) for w in (wg, wu, wd))
    href = orc.linear(synth.bf16_bits(x)[rows], og[0], og[1], og[2], wup=ou)
    assert_layer_close(bf16_to_f32(h)[rows], href, "dense gate/up")
    yref = orc.linear(synth.bf16_bits(torch.from_numpy(href).to(torch.bfloat16)), od[0], od[1], od[2])
    assert_layer_close(bf16_to_f32(y)[rows], yref, "dense down")


def test_linear_many_units_per_cta(orc):
    """Single-projection linear with 8192 rows, K=1536, N=4096: every CTA of
    the prompt-shaped kernel works through several (row tile, column slice)
    units, so ring slots are refilled many times; sampled rows from many
    tiles against the oracle."""
    M, K, N = 8192, 1536, 4096
    x = synth.make_x(M, K, seed=4101, device="cuda", outlier_frac=0.05)
    w = synth.make_weights(1, N, K, 4102, "cuda")[0]
    q = lib.nvfp4_quantize_weights(w)
    y = lib.nvfp4_linear(x, q)
    rows = np.unique(np.append(np.random.default_rng(4103).choice(M, 30, replace=False), [0, M - 1]))
    oq = orc.quantize_tensor(synth.bf16_bits(w))
    yref = orc.linear(synth.bf16_bits(x)[rows], oq[0], oq[1], oq[2])
    assert_layer_close(bf16_to_f32(y)[rows], yref, "linear K=1536 N=4096")


@pytest.mark.parametrize("T,E,k,d,F", [(512, 16, 4, 512, 256), (300, 6, 2, 1024, 384)])
def test_prompt_w4a4_tensor_cores(orc, T, E, k, d, F, monkeypatch):
    """W4A4 through the prompt-shaped tensor-core kernels (forced), several
    work units per expert, against the oracle on every token."""
    monkeypatch.setenv("NVFP4_PATH", "tc")
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob, r, tok = _setup(orc, s, seed=T + 7, outlier=0.05)
    xb = synth.bf16_bits(inp["x"])
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = lib.nvfp4_moe_w4a4(inp["x"], inp["logits"], k, gw, torch.from_numpy(is13).cuda(),
                             torch.from_numpy(is2).cuda(), d_status=st)
    ref = orc.moe_layer("w4a4", xb, r["ids"], r["w"], ob, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out), ref, "prompt w4a4")
    assert st[0].item() == 0


@pytest.mark.parametrize("mode", ["w4a16", "w4a4"])
def test_prompt_deterministic_and_chunk_invariant(orc, mode, monkeypatch):
    """The prompt-shaped path (forced) gives the same bits on every call and
    for any chunking of the batch: each routed row's result depends only on
    its own data (fixed K order, per-row scale), and each token's k weighted
    rows are summed in slot order."""
    monkeypatch.setenv("NVFP4_PATH", "tc")
    T, E, k, d, F = 512, 16, 4, 512, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob, r, tok = _setup(orc, s, seed=T + 23, outlier=0.05)
    x, lg = inp["x"], inp["logits"]
    if mode == "w4a16":
        run = lambda xx, ll: lib.nvfp4_moe_w4a16(xx, ll, k, gw)
    else:
        xb = synth.bf16_bits(x)
        is13, is2 = calib.calibrate(xb, lg.cpu().numpy(), k, ob)
        is13, is2 = torch.from_numpy(is13).cuda(), torch.from_numpy(is2).cuda()
        run = lambda xx, ll: lib.nvfp4_moe_w4a4(xx, ll, k, gw, is13, is2)
    full = run(x, lg)
    again = run(x, lg)
    assert torch.equal(full.view(torch.int16), again.view(torch.int16))
    parts = torch.cat([run(x[:200].contiguous(), lg[:200].contiguous()),
                       run(x[200:].contiguous(), lg[200:].contiguous())])
    assert torch.equal(full.view(torch.int16), parts.view(torch.int16))


@pytest.mark.parametrize("layer", [5, 30])
@pytest.mark.parametrize("kpath", ["gemv", "tc"])
def test_w4a4_layer_specific_calibration(orc, layer, kpath, monkeypatch):
    """W4A4 with the card's layer-specific w2 percentiles (p98 at layer 5,
    p98.9 at layer 30) on the decode and the prompt kernels, every token
    against the oracle."""
    monkeypatch.setenv("NVFP4_PATH", kpath)
    T, E, k, d, F = 256, 16, 4, 512, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp, gw, ob, r, tok = _setup(orc, s, seed=layer + 61, outlier=0.05)
    xb = synth.bf16_bits(inp["x"])
    p13, p2 = calib.layer_percentiles(layer)
    is13, is2 = calib.calibrate(xb, inp["logits"].cpu().numpy(), k, ob, pct13=p13, pct2=p2)
    out = lib.nvfp4_moe_w4a4(inp["x"], inp["logits"], k, gw, torch.from_numpy(is13).cuda(),
                             torch.from_numpy(is2).cuda())
    ref = orc.moe_layer("w4a4", xb, r["ids"], r["w"], ob, is13=is13, is2=is2)
    assert_layer_close(bf16_to_f32(out), ref, f"w4a4 layer {layer} {kpath}")
