"""The NVFP4 sublayer on the GPU against the oracle (itsolotime FlashRT
article, 7.2: norm + AWQ + FP4 quantise, gate and up NVFP4 GEMMs emitting
FP4, GeGLU FP4 -> FP4, NVFP4 down GEMM + residual).  Same inputs and scales on
both sides.  Contract: the block-scaled GEMM equals the exact sum within fp32
accumulation; weight preparation bit-exact; activation codes and block scales
identical wherever the oracle's value before rounding is not at a rounding
tie, E2M1 codes compared with +0 and -0 equal (FP4 values lie on a coarse
grid, so exact ties are common, and a last-ulp difference -- accumulation
order, the activation's hardware approximations -- may take the other side;
both roundings are valid there and must be one step apart), every step on
every row from the oracle's own input to it; layer outputs under the FP8
path's contract."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import bits, check_bf16, cosine

pytestmark = pytest.mark.gpu



# ---------------------------------------------------------------- layouts --

def pack(codes):
    """[rows, K] 4-bit codes -> [rows, K/2] bytes, element 2i in the low nibble."""
    c = np.asarray(codes, np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack(packed):
    p = np.asarray(packed, np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def _sf_index(rows, K):
    r = np.arange(rows)[:, None]
    g = np.arange(K // 16)[None, :]
    return ((r // 128) * (K // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4


def sf_to_tmem(sf):
    """Row-major block scales [rows, K/16] -> the TMEM-ready layout (rows padded to 128)."""
    sf = np.asarray(sf, np.uint8)
    rows, G = sf.shape
    K = G * 16
    out = np.zeros(((rows + 127) // 128) * 128 * G, np.uint8)
    out[_sf_index(rows, K)] = sf
    return out


def sf_from_tmem(buf, rows, K):
    return np.asarray(buf, np.uint8)[_sf_index(rows, K)]


def canon(codes):
    """E2M1 codes with -0 (8) read as +0."""
    c = np.asarray(codes, np.uint8)
    return np.where(c == 8, 0, c).astype(np.uint8)


def ordinal(codes):
    c = canon(codes).astype(np.int32)
    return np.where(c & 8, -(c & 7), c & 7)


E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_E4M3_POS = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
E4M3_MIDS = (_E4M3_POS[:-1] + _E4M3_POS[1:]) / 2
TIE_REL = 2e-3  # two fp32 evaluations of the same value (accumulation order, tanhf ulps) differ far less


def near_tie(t, mids):
    """|t| within TIE_REL of a rounding midpoint (where either rounding is valid)."""
    t = np.abs(np.asarray(t, np.float64)).ravel()
    if t.size == 0:
        return np.zeros(0, bool)
    d = np.abs(t[:, None] - mids[None, :]).min(axis=1)
    return d <= TIE_REL * np.maximum(t, 1e-30)


def check_nvfp4(got_q, got_sb, ref_q, ref_sb, x, s, what):
    """GPU NVFP4 codes and block scales against the oracle's: identical except
    where the oracle's own pre-rounding value sits at a rounding tie (block
    scale: amax / (6 s) at an E4M3 midpoint; element: x / (dec(b) s) at an
    E2M1 midpoint), and then one step apart.  x: the oracle's fp32 values
    before quantisation [rows, K]."""
    x = np.asarray(x, np.float32)
    rows, K = x.shape
    blk = x.reshape(rows, K // 16, 16)
    inv6 = np.float32(oracle.recip(np.float32(6.0) * np.float32(s)))
    t_sb = (np.abs(blk).max(axis=2) * inv6).astype(np.float32)
    gsb, rsb = np.asarray(got_sb, np.int32), np.asarray(ref_sb, np.int32)
    dsb = gsb != rsb
    assert np.abs(gsb - rsb).max(initial=0) <= 1, "%s: block scales more than one step apart" % what
    assert near_tie(t_sb[dsb], E4M3_MIDS).all(), "%s: a block scale differs off a rounding tie" % what
    assert dsb.mean() <= 0.01, "%s: %.4f of block scales differ" % (what, dsb.mean())
    den = (oracle.e4m3_decode(np.asarray(ref_sb, np.uint8)) * np.float32(s)).astype(np.float32)
    inv = np.where(den > 0, np.float32(1) / np.where(den > 0, den, 1), 0).astype(np.float32)
    t_q = (blk * inv[:, :, None]).astype(np.float32).reshape(rows, K)
    g, r = ordinal(got_q), ordinal(ref_q)
    same_blk = np.repeat(~dsb, 16, axis=1)
    dq = (g != r) & same_blk
    assert np.abs(g - r)[same_blk].max(initial=0) <= 1, "%s: E2M1 codes more than one step apart" % what
    assert near_tie(t_q[dq], E2M1_MIDS).all(), "%s: an E2M1 code differs off a rounding tie" % what
    assert dq.mean() <= 0.01, "%s: %.4f of E2M1 codes differ" % (what, dq.mean())
    return ~(dsb.any(axis=1) | (g != r).any(axis=1))


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------- GEMM --

@pytest.mark.parametrize("swap", [False, True], ids=["tiled", "weight_streaming"])
@pytest.mark.parametrize("M,N,K,S", [(1, 128, 256, 1), (50, 256, 512, 1), (128, 128, 2048, 1), (300, 384, 1024, 1),
                                     (1, 256, 2048, 3), (50, 128, 4096, 8), (300, 256, 1024, 2),
                                     (256, 256, 1024, 1), (500, 384, 512, 2)])
def test_block_scaled_gemm_matches_the_exact_sum(M, N, K, S, swap, monkeypatch):
    from realtime_transformer_gb300.nvfp4 import nvfp4_gemm
    if swap and M > 64:
        pytest.skip("the weight-streaming role takes at most 64 tokens")
    monkeypatch.setenv("FRT_F4_SWAP", "1" if swap else "0")
    rng = np.random.default_rng(M * 7 + N + K)
    qa = rng.integers(0, 16, (M, K)).astype(np.uint8)
    qb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = rng.integers(0x28, 0x48, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0x28, 0x48, (N, K // 16)).astype(np.uint8)
    alpha = 0.375
    out, err, _ = nvfp4_gemm(dev(pack(qa)), dev(sf_to_tmem(sa)), dev(pack(qb)), dev(sf_to_tmem(sb)), M, N, K,
                             alpha, splits=S)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = (oracle.nvfp4_gemm(qa, sa, qb, sb).astype(np.float64) * alpha)
    got = out.cpu().numpy().astype(np.float64)
    rms = np.sqrt((ref ** 2).mean())
    assert np.abs(got - ref).max() <= 1e-5 * rms * np.sqrt(K), (np.abs(got - ref).max(), rms)
    assert cosine(got, ref) > 0.9999999


# "1": the weight-streaming role; "0": the tiled role (130, 256: several token
# tiles; N = 256: 256-row weight tiles, whose second 128 rows have scale
# columns of their own)
@pytest.mark.parametrize("M,swap,N", [(130, "0", 128), (256, "0", 128), (40, "0", 128), (40, "1", 128),
                                      (130, "0", 256), (40, "1", 256)])
def test_gemm_scale_placement_one_block_at_a_time(M, swap, N, monkeypatch):
    """Only one (row, K-group) scale of A nonzero: the product picks exactly
    that row's 16 elements of K -- pins the TMEM-ready layout end to end."""
    from realtime_transformer_gb300.nvfp4 import nvfp4_gemm
    monkeypatch.setenv("FRT_F4_SWAP", swap)
    K = 512
    rng = np.random.default_rng(9)
    qa = rng.integers(0, 16, (M, K)).astype(np.uint8)
    qb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sb = np.full((N, K // 16), 0x38, np.uint8)  # 1.0
    for (m, g) in [(0, 0), (37, 5), (99, 31), (129, 17)]:
        if m >= M:
            continue
        sa = np.zeros((M, K // 16), np.uint8)
        sa[m, g] = 0x38
        out, err, _ = nvfp4_gemm(dev(pack(qa)), dev(sf_to_tmem(sa)), dev(pack(qb)), dev(sf_to_tmem(sb)), M, N, K,
                                 splits=2)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref = oracle.nvfp4_gemm(qa, sa, qb, sb)
        assert np.array_equal(got, ref), (m, g)
        assert np.count_nonzero(got[np.arange(M) != m]) == 0
    sa = np.full((M, K // 16), 0x38, np.uint8)
    for (n, g) in [(0, 3), (64, 12), (127, 30), (128, 1), (200, 22), (255, 31)]:
        if n >= N:
            continue
        sb = np.zeros((N, K // 16), np.uint8)
        sb[n, g] = 0x38
        out, err, _ = nvfp4_gemm(dev(pack(qa)), dev(sf_to_tmem(sa)), dev(pack(qb)), dev(sf_to_tmem(sb)), M, N, K,
                                 splits=2)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got, oracle.nvfp4_gemm(qa, sa, qb, sb)), (n, g)
        assert np.count_nonzero(got[:, np.arange(N) != n]) == 0


# ------------------------------------------------------------ the sublayer --

CASES = {
    "tiny": synthetic.WORKLOADS["tiny"],
    "action_expert": synthetic.WORKLOADS["vla_action_expert"].with_(L=1),
    "ragged": synthetic.WORKLOADS["tiny"].with_(name="ragged", M=300, d=512, ff=1024, act="swiglu", seed=5),
    # one token, as decode: the weight-streaming role's 16-token tile with 15 padding rows
    "m1_swiglu": synthetic.WORKLOADS["tiny"].with_(name="m1_swiglu", M=1, d=1024, ff=2048, act="swiglu", seed=6),
}


def _awq_for(wl, lw):
    cb = synthetic.calibration_batches(wl)
    ys = [oracle.residual_rmsnorm(bits(a), bits(b), bits(lw["w_norm"]))[1] for a, b in cb]
    return oracle.awq_scales(ys, 0.5)


@pytest.fixture(scope="module", params=[(k, a) for k in CASES for a in (False, True) if k != "ragged" or not a],
                ids=lambda p: p[0] + ("_awq" if p[1] else ""))
def layer_case(request):
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    name, use_awq = request.param
    wl = CASES[name]
    lw = synthetic.layer_weights(wl, 0)
    r, h = synthetic.inputs(wl)
    cb = synthetic.calibration_batches(wl)
    awq = _awq_for(wl, lw) if use_awq else None
    L = oracle.quantize_layer_nvfp4(bits(lw["w_norm"]), bits(lw["w_gate"]), bits(lw["w_up"]), bits(lw["w_down"]),
                                    awq)
    sc, _ = oracle.calibrate_layer_nvfp4([bits(a) for a, _ in cb], [bits(b) for _, b in cb], L, wl.act_id)
    plan = FP4Plan(wl.d, wl.ff, wl.act, wl.M, 1)
    plan.load_weights(0, *(lw[k].cuda() for k in ("w_norm", "w_gate", "w_up", "w_down")),
                      awq=dev(awq) if awq is not None else None)
    plan.set_scales([[sc.s_x, sc.s_g, sc.s_u, sc.s_h]])
    yield dict(wl=wl, lw=lw, r=r, h=h, L=L, sc=sc, plan=plan, cb=cb)
    plan.close()


def test_weight_preparation_is_bit_exact(layer_case):
    c = layer_case
    wl, L, plan = c["wl"], c["L"], c["plan"]
    s_w = plan.scales()["weight"][0]
    for which, ref, rows, K, s in [("gate", L.gate, wl.ff, wl.d, s_w[0]), ("up", L.up, wl.ff, wl.d, s_w[1]),
                                   ("down", L.down, wl.d, wl.ff, s_w[2])]:
        codes, sf = plan.weights(0, which)
        assert np.float32(s) == np.float32(ref.s), which
        assert np.array_equal(canon(unpack(codes.cpu().numpy())), canon(ref.q)), which
        assert np.array_equal(sf_from_tmem(sf.cpu().numpy(), rows, K), ref.sb), which


def test_layer_matches_oracle(layer_case):
    """Every step on every row, each started from the oracle's own input to
    that step (the GPU GEMMs fed the oracle's X and A through
    frt_fp4_debug_trace_from; the combine checked on the GPU's own G and U);
    then the kernels' own path through the whole layer."""
    c = layer_case
    wl, plan, sc = c["wl"], c["plan"], c["sc"]
    r, h = c["r"].cuda(), c["h"].cuda()
    ref = oracle.ffn_layer_nvfp4(bits(c["r"]), bits(c["h"]), c["L"], sc, wl.act_id, trace=True)
    M, d, ff = wl.M, wl.d, wl.ff
    tr = plan.trace(0, r, h)
    torch.cuda.synchronize()
    plan.device_status()
    # N1: r' bit for bit, X under the tie-aware code contract
    assert np.array_equal(bits(tr["r_prime"]), ref.r_prime)
    check_nvfp4(unpack(tr["x_codes"].cpu().numpy()), sf_from_tmem(tr["x_sf"].cpu().numpy(), M, d), ref.x[0],
                ref.x[1], ref.y, sc.s_x, "x")
    tf = plan.trace_from(0, r, h, x=(dev(pack(ref.x[0])), dev(sf_to_tmem(ref.x[1]))),
                         h=(dev(pack(ref.h[0])), dev(sf_to_tmem(ref.h[1]))))
    torch.cuda.synchronize()
    plan.device_status()
    # N2 from the oracle's X: G and U
    gq, gs = unpack(tf["g_codes"].cpu().numpy()), tf["g_sf"].cpu().numpy()
    uq, us = unpack(tf["u_codes"].cpu().numpy()), tf["u_sf"].cpu().numpy()
    check_nvfp4(gq, gs, ref.g[0], ref.g[1], ref.g_f32, sc.s_g, "gate")
    check_nvfp4(uq, us, ref.u[0], ref.u[1], ref.u_f32, sc.s_u, "up")
    # N3 on the GPU's own G and U: the oracle's combine of those codes
    a = oracle.nvfp4_gated_act((gq, gs), (uq, us), sc.s_g, sc.s_u, wl.act_id)
    h_ref = oracle.nvfp4_quantize(a, sc.s_h)
    check_nvfp4(unpack(tf["h_codes"].cpu().numpy()), sf_from_tmem(tf["h_sf"].cpu().numpy(), M, ff), h_ref[0],
                h_ref[1], a, sc.s_h, "h")
    # N4 from the oracle's A: the output under the FP8 path's contract
    check_bf16(bits(tf["out"]), ref.out, "out")
    # the kernels' own path through the layer
    got_all = oracle.bf16_decode(bits(tr["out"]))
    assert cosine(got_all, oracle.bf16_decode(ref.out)) > 0.9999
    # the stack entry point (one layer) computes what the trace computes
    o = plan.forward(r, h)
    torch.cuda.synchronize()
    assert torch.equal(o, tr["out"])


def test_weight_streaming_role_matches_the_tiled_role(layer_case, monkeypatch):
    """At most 64 tokens: the weight-streaming role computes the same layer
    (same quantised activations except at rounding ties of the sums)."""
    c = layer_case
    if c["wl"].M > 64:
        pytest.skip("the weight-streaming role takes at most 64 tokens")
    r, h = c["r"].cuda(), c["h"].cuda()
    monkeypatch.setenv("FRT_F4_SWAP", "0")
    a = c["plan"].trace(0, r, h)
    monkeypatch.setenv("FRT_F4_SWAP", "1")
    b = c["plan"].trace(0, r, h)
    torch.cuda.synchronize()
    assert torch.equal(a["x_codes"], b["x_codes"]) and torch.equal(a["x_sf"], b["x_sf"])
    for k in ("g_codes", "u_codes", "h_codes"):
        same = float((a[k] == b[k]).float().mean())
        assert same > 0.99, (k, same)
    assert cosine(oracle.bf16_decode(bits(a["out"])), oracle.bf16_decode(bits(b["out"]))) > 0.9999


def test_forward_can_be_captured_in_a_cuda_graph(layer_case):
    c = layer_case
    plan = c["plan"]
    r, h = c["r"].cuda(), c["h"].cuda()
    eager = plan.forward(r, h)
    torch.cuda.synchronize()
    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.forward(r, h, out=out, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            plan.forward(r, h, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_forward_profile_splits_the_stack_and_computes_the_forward():
    """The stamped replays: one share per launch (3 per layer), each positive,
    together at most the replay's span; the profiled graph writes the same
    output as the eager forward."""
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    wl = synthetic.WORKLOADS["tiny"].with_(L=3, M=40)
    plan = FP4Plan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    try:
        for l in range(wl.L):
            w = synthetic.layer_weights(wl, l, device=torch.device("cuda"))
            plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"])
        plan.set_scales([[0.02, 0.05, 0.05, 0.01]] * wl.L)
        r, h = (t.cuda() for t in synthetic.inputs(wl))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            eager = plan.forward(r, h, stream=s)
            s.synchronize()
            out = torch.zeros_like(eager)
            shares = plan.forward_profile(r, h, out=out, n_replays=5, stream=s)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(10):
                plan.forward(r, h, out=out, stream=s)
            e1.record(s)
        s.synchronize()
        assert torch.equal(out, eager)
        assert len(shares) == 3 * wl.L
        assert all(x > 0.0 for x in shares), shares
        # the eager forward's time bounds the replayed graph's stamped span
        assert sum(shares) <= e0.elapsed_time(e1) * 1000.0 / 10 + 5.0, (sum(shares), shares)
        with pytest.raises(Exception):
            plan.forward_profile(r, h, out=out, n_replays=0, stream=s)
    finally:
        plan.close()


def test_gpu_calibration_and_stack_match_oracle():
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    wl = synthetic.WORKLOADS["tiny"].with_(L=3, M=40)
    layers = [synthetic.layer_weights(wl, l) for l in range(wl.L)]
    r, h = synthetic.inputs(wl)
    cb = synthetic.calibration_batches(wl)
    Ls = [oracle.quantize_layer_nvfp4(*(bits(lw[k]) for k in ("w_norm", "w_gate", "w_up", "w_down")))
          for lw in layers]
    ref_sc = oracle.calibrate_stack_nvfp4(Ls, [bits(a) for a, _ in cb], [bits(b) for _, b in cb], wl.act_id)
    plan = FP4Plan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    try:
        for l, lw in enumerate(layers):
            plan.load_weights(l, *(lw[k].cuda() for k in ("w_norm", "w_gate", "w_up", "w_down")))
        plan.calibrate([a.cuda() for a, _ in cb], [b.cuda() for _, b in cb])
        got = plan.scales()["act"]
        for l in range(wl.L):
            want = [ref_sc[l].s_x, ref_sc[l].s_g, ref_sc[l].s_u, ref_sc[l].s_h]
            # s_x, s_g, s_u: amax of fp32 tensors both sides compute alike; s_h
            # follows E2M1 codes that may take the other valid rounding
            for i, tol in enumerate((1e-5, 1e-4, 1e-4, 5e-2)):
                assert abs(got[l][i] - want[i]) <= tol * want[i], (l, i, got[l][i], want[i])
        out = plan.forward(r.cuda(), h.cuda())
        torch.cuda.synchronize()
        plan.device_status()
        ref = oracle.stack_forward_nvfp4(Ls, ref_sc, bits(r), bits(h), wl.act_id)
        assert cosine(oracle.bf16_decode(bits(out)), oracle.bf16_decode(ref)) > 0.9999
    finally:
        plan.close()


def test_boundary_errors():
    from realtime_transformer_gb300 import _native as N
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    p = FP4Plan(256, 512, "swiglu", 8, 2)
    r = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(N.FrtError) as e:
        p.forward(r)
    assert e.value.name == "FRT_ERR_NOT_READY"
    w = synthetic.layer_weights(synthetic.WORKLOADS["tiny"].with_(d=256, ff=512), 0)
    for l in range(2):
        p.load_weights(l, *(w[k].cuda() for k in ("w_norm", "w_gate", "w_up", "w_down")))
    with pytest.raises(N.FrtError) as e:
        p.forward(r)  # no activation scales yet
    assert e.value.name == "FRT_ERR_NOT_READY"
    with pytest.raises(N.FrtError) as e:
        p.set_scales([[0.01, 0.01, 0.01, 0.01], [0.01, float("nan"), 0.01, 0.01]])
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    with pytest.raises(N.FrtError) as e:
        p.load_weights(0, *(w[k].cuda() for k in ("w_norm", "w_gate", "w_up", "w_down")),
                       awq=-torch.ones(256, device="cuda"))
    assert e.value.name == "FRT_ERR_INVALID_ARG"
    p.set_scales([[0.01] * 4, [0.01] * 4])
    big = torch.zeros(9, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(N.FrtError) as e:
        p.forward(big)
    assert e.value.name == "FRT_ERR_SHAPE"
    N.frt_fp4_forward(p.handle, r.data_ptr(), None, torch.empty_like(r).data_ptr(), 0, None)  # M == 0: nothing
    p.device_status()
    p.close()
