"""Pins of the fp64 oracle against things other than itself.

Each test ties one part of the oracle to a hand-derived example, a closed form,
a library routine on a special case, an invariant or brute force, chosen so
that a plausible slip (dropped bias, unnormalised g, swapped up/gate,
transposed operand, wrong expert index, wrong tie-break or slot order, wrong
schedule position, wrong MX scale or rounding) fails at least one of them.
Sources: "Mixture-of-Kittens: MoE Megakernel for NVL72s" Sec. 2.1 (Eq. MoE),
Sec. 3.1 (Algorithm 1 and its sort-key reading), Sec. 3.4 (MXFP8); the vendor
blog's MoE(x,s) / E_i(x) formulas (SiLU).
"""
import math
import random

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle


def f64(bits):
    return mi.bf16_bits_to_f32(bits).astype(np.float64)


def dense_ffn(x, w_up, w_gate, w_down):
    """W_down (SiLU(W_gate x) * W_up x) for rows of x, by numpy fp64 matmuls."""
    u = x @ w_up.T
    v = x @ w_gate.T
    h = v / (1.0 + np.exp(-v)) * u
    return h @ w_down.T


def small_inputs(T=40, D=64, I=32, E=8, k=3, I_s=32, score="sigmoid", cid=200, beta=True):
    shape = mi.custom_shape(T, D, I, E, k, I_s, score=score, config_id=cid)
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    if beta:
        inp.b_router = (0.25 * mi.normal_f64(shape.seed, 99, E)).astype(np.float32)
    return inp


# ------------------------------------------------------------------ hand examples
def test_topk_hand_examples(golden):
    for ex in golden["topk"]:
        lg = np.array([ex["logits"]])
        idx, g = oracle.topk(lg, ex["k"], ex["score"])
        assert idx[0].tolist() == ex["idx"], ex["why"]
        np.testing.assert_allclose(g[0], ex["g"], rtol=1e-14, atol=0)


def test_scalar_ffn_hand_example(golden):
    ex = golden["ffn_scalar"]
    shape = mi.custom_shape(1, 1, 1, 1, 1, 0)
    b = lambda v: mi.f32_to_bf16_bits(np.array([[v]], dtype=np.float32))
    out, idx, g = oracle.moe_fwd(shape, b(ex["x"]), b(1.0), None, b(ex["w_up"])[None], b(ex["w_gate"])[None],
                                 b(ex["w_down"])[None])
    assert idx[0, 0] == 0 and g[0, 0] == 1.0
    assert out[0, 0] == pytest.approx(ex["y"], rel=1e-14)


# ------------------------------------------------------------------ router / top-k
@pytest.mark.parametrize("score", ["sigmoid", "softmax"])
def test_router_logits_match_numpy_matmul(score):
    inp = small_inputs(score=score)
    lg = oracle.router_logits(inp.x, inp.w_router, inp.b_router)
    ref = f64(inp.x) @ f64(inp.w_router).T + inp.b_router.astype(np.float64)
    np.testing.assert_allclose(lg, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("score,k,E", [("sigmoid", 3, 8), ("softmax", 4, 16), ("sigmoid", 1, 5), ("sigmoid", 6, 6)])
def test_topk_brute_force(score, k, E):
    """Both score functions are increasing in the logit, so the top-k by score
    is the top-k by logit: brute-force sort of (-logit, id), then ascending id."""
    rng = np.random.default_rng(7 + k)
    lg = rng.normal(size=(300, E))
    lg[:20, :] = np.round(lg[:20, :])  # exact ties exercise the lower-id rule
    idx, g = oracle.topk(lg, k, score)
    for t in range(lg.shape[0]):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))
        assert idx[t].tolist() == sorted(order[:k])


def test_g_sums_to_one():
    inp = small_inputs()
    _, _, g = oracle.moe_fwd_inputs(inp)
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=0, atol=1e-12)


def test_softmax_g_closed_form():
    """g_i = s_i / sum_sel s_j with s = softmax over all E; the normaliser
    cancels, leaving exp(l_i) / sum_sel exp(l_j)."""
    rng = np.random.default_rng(3)
    lg = rng.normal(size=(50, 12)) * 2
    idx, g = oracle.topk(lg, 4, "softmax")
    for t in range(50):
        sel = lg[t, idx[t]]
        want = [math.exp(v) / sum(math.exp(w) for w in sel) for v in sel]
        np.testing.assert_allclose(g[t], want, rtol=1e-13)


def test_bias_changes_selection():
    """A large bias on one expert must put it into every token's top-k."""
    inp = small_inputs(beta=False)
    inp.b_router = np.zeros(inp.shape.E, dtype=np.float32)
    inp.b_router[5] = 50.0
    _, idx, _ = oracle.moe_fwd_inputs(inp)
    assert (idx == 5).any(axis=1).all()


# ------------------------------------------------------------------ layer special cases
def test_one_expert_top1_is_dense_ffn():
    """E = 1, k = 1, no shared expert: MoE(x) = f(x) exactly (g = 1)."""
    inp = small_inputs(E=1, k=1, I_s=0, D=96, I=40)
    out, _, g = oracle.moe_fwd_inputs(inp)
    assert (g == 1.0).all()
    ref = dense_ffn(f64(inp.x), f64(inp.w_up[0]), f64(inp.w_gate[0]), f64(inp.w_down[0]))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_top1_uses_the_selected_experts_weights():
    """k = 1 with many experts: out = f_shared(x) + f_{argmax}(x), each term by numpy."""
    inp = small_inputs(E=8, k=1, I_s=24, D=64, I=40)
    out, idx, _ = oracle.moe_fwd_inputs(inp)
    xf = f64(inp.x)
    shared = dense_ffn(xf, f64(inp.ws_up), f64(inp.ws_gate), f64(inp.ws_down))
    for t in range(xf.shape[0]):
        e = idx[t, 0]
        ref = shared[t] + dense_ffn(xf[t:t + 1], f64(inp.w_up[e]), f64(inp.w_gate[e]), f64(inp.w_down[e]))[0]
        np.testing.assert_allclose(out[t], ref, rtol=1e-11, atol=1e-12)
    lg = f64(inp.x) @ f64(inp.w_router).T + inp.b_router
    assert (idx[:, 0] == lg.argmax(1)).all()


def test_identical_experts_collapse():
    """All routed experts equal: sum g = 1 gives MoE(x) = f_shared(x) + f(x)."""
    inp = small_inputs(E=6, k=3)
    for w in (inp.w_up, inp.w_gate, inp.w_down):
        w[:] = w[0]
    out, _, _ = oracle.moe_fwd_inputs(inp)
    xf = f64(inp.x)
    ref = dense_ffn(xf, f64(inp.ws_up), f64(inp.ws_gate), f64(inp.ws_down)) + \
        dense_ffn(xf, f64(inp.w_up[0]), f64(inp.w_gate[0]), f64(inp.w_down[0]))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_scaled_down_projections_weight_by_g():
    """W_up, W_gate shared by all experts and W_down^(e) = c_e W0 (powers of two,
    exact in bf16): MoE(x) - f_shared(x) = (sum_i g_i c_i) f0(x)."""
    inp = small_inputs(E=8, k=3)
    c = np.array([2.0 ** ((e % 5) - 2) for e in range(8)])
    inp.w_up[:] = inp.w_up[0]
    inp.w_gate[:] = inp.w_gate[0]
    w0 = f64(inp.w_down[0])
    for e in range(8):
        inp.w_down[e] = mi.f32_to_bf16_bits((w0 * c[e]).astype(np.float32))
    out, idx, g = oracle.moe_fwd_inputs(inp)
    xf = f64(inp.x)
    shared = dense_ffn(xf, f64(inp.ws_up), f64(inp.ws_gate), f64(inp.ws_down))
    f0 = dense_ffn(xf, f64(inp.w_up[0]), f64(inp.w_gate[0]), w0)
    coef = (g * c[idx]).sum(1)
    np.testing.assert_allclose(out - shared, coef[:, None] * f0, rtol=1e-10, atol=1e-12)


def test_zero_shared_expert_removes_exactly_the_shared_term():
    inp = small_inputs()
    with_shared, _, _ = oracle.moe_fwd_inputs(inp)
    z = small_inputs()
    z.ws_up = np.zeros_like(z.ws_up)
    z.ws_gate = np.zeros_like(z.ws_gate)
    z.ws_down = np.zeros_like(z.ws_down)
    zeroed, _, _ = oracle.moe_fwd_inputs(z)
    n = small_inputs()
    n.ws_up = n.ws_gate = n.ws_down = None
    without, _, _ = oracle.moe_fwd_inputs(n)
    assert np.array_equal(zeroed, without)  # bitwise
    shared = dense_ffn(f64(inp.x), f64(inp.ws_up), f64(inp.ws_gate), f64(inp.ws_down))
    np.testing.assert_allclose(with_shared - without, shared, rtol=1e-9, atol=1e-12)


def test_down_projection_linearity_bitwise():
    """Doubling every W_down (exact in bf16) doubles the routed output exactly."""
    a = small_inputs(I_s=0)
    b = small_inputs(I_s=0)
    b.w_down = mi.f32_to_bf16_bits(mi.bf16_bits_to_f32(b.w_down) * 2.0).reshape(b.w_down.shape)
    oa, _, _ = oracle.moe_fwd_inputs(a)
    ob, _, _ = oracle.moe_fwd_inputs(b)
    assert np.array_equal(ob, 2.0 * oa)


def test_token_permutation_equivariance():
    inp = small_inputs(T=33)
    out, idx, g = oracle.moe_fwd_inputs(inp)
    perm = np.random.default_rng(5).permutation(33)
    outp, idxp, gp = oracle.moe_fwd_inputs(inp, rows=perm)
    assert np.array_equal(outp, out[perm]) and np.array_equal(idxp, idx[perm]) and np.array_equal(gp, g[perm])


def test_token_subset_equals_full_run():
    """Tokens are independent: a subset run gives the same bits as the full run."""
    inp = small_inputs(T=50)
    out, idx, _ = oracle.moe_fwd_inputs(inp)
    rows = np.array([49, 0, 17, 17, 3])
    o2, i2, _ = oracle.moe_fwd_inputs(inp, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(i2, idx[rows])


# ------------------------------------------------------------------ schedule (Algorithm 1)
@pytest.mark.parametrize("R,L,N,K,c", [(1, 4, 10, 2, 0), (2, 3, 7, 2, 1), (3, 2, 9, 3, 0), (3, 4, 5, 4, 2)])
def test_alg1_round_robin_merge_equals_sort_key(R, L, N, K, c):
    """Sec. 3.1: the table is the routes sorted by (local expert, ordinal o,
    source rank r); the count-scan-merge construction must produce exactly it."""
    rnd = random.Random(R * 100 + L * 10 + N)
    for _ in range(20):
        A = []
        for _r in range(R):
            routes = []
            for _t in range(N):
                routes += rnd.sample(range(R * L), K)
            A.append(routes)
        phi, M, S = oracle.alg1_schedule(A, c, L)
        assert phi == oracle.sort_key_schedule(A, c, L)
        assert None not in phi
        # round-robin interleave: within an expert region, consecutive entries
        # with the same ordinal come from increasing ranks
        assert sorted(phi) == sorted(set(phi))


def test_single_rank_schedule_matches_alg1_and_stable_argsort():
    inp = small_inputs(T=64, E=8, k=3)
    _, idx, _ = oracle.moe_fwd_inputs(inp)
    M, S, sched, route_row = oracle.schedule(idx, 8)
    flat = idx.reshape(-1)
    # numpy stable argsort by expert id is the permutation (library routine)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(sched[:, 2], order)
    assert np.array_equal(sched[:, 1], flat[order])
    assert np.array_equal(sched[:, 0], order // 3)
    assert np.array_equal(route_row[order], np.arange(flat.size))
    assert np.array_equal(M, np.bincount(flat, minlength=8))
    assert S[0] == 0 and np.array_equal(np.diff(S), M)
    # pure-Python Algorithm 1 with R = 1
    phi, M1, S1 = oracle.alg1_schedule([flat.tolist()], 0, 8)
    assert [j for (_r, j) in phi] == sched[:, 2].tolist()


def test_schedule_invariants_and_empty_experts():
    idx = np.array([[0, 5], [0, 5], [2, 5]], dtype=np.int32)
    M, S, sched, route_row = oracle.schedule(idx, 7)
    assert M.tolist() == [2, 0, 1, 0, 0, 3, 0]
    assert S.tolist() == [0, 2, 2, 3, 3, 3, 6, 6]
    assert sched.tolist() == [[0, 0, 0], [1, 0, 2], [2, 2, 4], [0, 5, 1], [1, 5, 3], [2, 5, 5]]
    assert route_row.tolist() == [0, 3, 1, 4, 2, 5]
    with pytest.raises(ValueError):
        oracle.schedule(np.array([[7]], dtype=np.int32), 7)


# ------------------------------------------------------------------ MXFP8
def test_mx_hand_examples(golden):
    for key in ("mx_block", "mx_saturation"):
        ex = golden[key]
        v = np.zeros((1, 32))
        v[0, :len(ex["values_head"])] = ex["values_head"]
        q, s = oracle.mx_quantize(v)
        assert s[0, 0] == ex["scale_code"], ex["why"]
        assert q[0, :len(ex["codes_head"])].tolist() == ex["codes_head"], ex["why"]
        if "dequant_head" in ex:
            dq = oracle.mx_dequantize(q, s)
            assert dq[0, :4].tolist() == ex["dequant_head"]


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_rounding():
    """Round-to-nearest-even on in-range values, compared with torch's
    float32 -> float8_e4m3fn conversion (halfway cases included)."""
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.normal(size=4000) * 50, rng.normal(size=2000) * 0.01,
                           np.array([2.0 ** -10, 3 * 2.0 ** -10, 0.5 * 2.0 ** -9, 1.5 * 2.0 ** -9, 448.0, -448.0,
                                     17.0, 19.0, 0.0])]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    # +0 and -0 both mean zero
    ref = np.where((ref & 0x7F) == 0, 0, ref)
    mine = np.where((mine & 0x7F) == 0, 0, mine)
    assert np.array_equal(mine, ref)


def test_mx_scale_rule_and_error_bound():
    rng = np.random.default_rng(12)
    v = rng.normal(size=(64, 96)) * np.exp(rng.normal(size=(64, 1)) * 4)
    q, s = oracle.mx_quantize(v)
    dq = oracle.mx_dequantize(q, s)
    for r in range(64):
        for b in range(3):
            blk = v[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            m, e = math.frexp(amax)
            assert s[r, b] == (e - 1) - 8 + 127  # X = 2^(floor(log2 amax) - 8)
            X = 2.0 ** (int(s[r, b]) - 127)
            assert 256.0 <= amax / X < 512.0
    assert np.abs(oracle.mx_dequantize(q, s)).max() <= 448.0 * 2.0 ** (int(s.max()) - 127)
    # relative error of unsaturated normal elements <= 2^-4 (3 mantissa bits)
    X = 2.0 ** (s.astype(np.float64) - 127).repeat(32, axis=1)
    scaled = np.abs(v) / X
    normal = (scaled >= 2.0 ** -6) & (scaled <= 448.0)
    rel = np.abs(dq - v)[normal] / np.abs(v)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-15


def test_mx_roundtrip_of_representable_values():
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 256, size=(16, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10  # no NaN codes
    codes[:, 0] = 0x78  # one element of magnitude 256 per block makes the block max exact
    codes[:, 32] = 0xF8
    scales = rng.integers(100, 140, size=(16, 2)).astype(np.uint8)
    v = oracle.mx_dequantize(codes, scales)
    q, s = oracle.mx_quantize(v)
    assert np.array_equal(oracle.mx_dequantize(q, s), v)
    assert np.array_equal(s, scales)


def test_mx_zero_block():
    q, s = oracle.mx_quantize(np.zeros((2, 64)))
    assert (q == 0).all() and (s == 0).all()


def test_mx_bf16_input_path_equals_f64_path():
    rng = np.random.default_rng(14)
    bits = mi.f32_to_bf16_bits(rng.normal(size=(8, 64)).astype(np.float32))
    q1, s1 = oracle.mx_quantize(bits)
    q2, s2 = oracle.mx_quantize(f64(bits))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_mx_layer_dense_special_case():
    """E = 1, k = 1, no shared expert, MX experts: out = W_down' q(h) with
    h = SiLU(W_gate' q(x)) * W_up' q(x); W' the dequantised weights, q the MX
    round trip (pinned above); the matmuls by numpy."""
    inp = small_inputs(E=1, k=1, I_s=0, D=64, I=64)
    mx = {}
    for name, w in (("up", inp.w_up), ("gate", inp.w_gate), ("down", inp.w_down)):
        mx[name + "_q"], mx[name + "_s"] = oracle.mx_quantize(w)
    out, _, _ = oracle.moe_fwd_inputs(inp, mx=mx)
    deq = {n: oracle.mx_dequantize(mx[n + "_q"], mx[n + "_s"])[0] for n in ("up", "gate", "down")}
    xq = oracle.mx_dequantize(*oracle.mx_quantize(f64(inp.x)))
    u = xq @ deq["up"].T
    v = xq @ deq["gate"].T
    h = v / (1.0 + np.exp(-v)) * u
    hq = oracle.mx_dequantize(*oracle.mx_quantize(h))
    np.testing.assert_allclose(out, hq @ deq["down"].T, rtol=1e-9, atol=1e-12)


def test_mx_layer_close_to_bf16_layer():
    inp = small_inputs(E=8, k=2, I_s=32, D=128, I=64, T=64)
    mx = {}
    for name, w in (("up", inp.w_up), ("gate", inp.w_gate), ("down", inp.w_down)):
        mx[name + "_q"], mx[name + "_s"] = oracle.mx_quantize(w)
    out_mx, idx_mx, _ = oracle.moe_fwd_inputs(inp, mx=mx)
    out, idx, _ = oracle.moe_fwd_inputs(inp)
    assert np.array_equal(idx, idx_mx)  # the router is not quantised
    rel = np.linalg.norm(out_mx - out) / np.linalg.norm(out)
    assert 1e-4 < rel < 6e-2


# ------------------------------------------------------------------ input generator
def test_generator_is_deterministic_and_standard_normal():
    a = mi.normal_f64(123, 1, 200000)
    b = mi.normal_f64(123, 1, 200000)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.01 and abs(a.var() - 1) < 0.01
    c = mi.normal_f64(123, 1, 1000, start=500)
    assert np.array_equal(c, a[500:1500])
    bits = mi.normal_bf16(123, 1, 1000)
    assert np.array_equal(bits, mi.f32_to_bf16_bits(a[:1000].astype(np.float32)))


def test_redrawn_rows_use_their_own_stream():
    att = np.zeros(10, dtype=np.int32)
    x0 = mi.x_rows(5, 10, 32, att)
    att[3] = 1
    x1 = mi.x_rows(5, 10, 32, att)
    assert np.array_equal(np.delete(x0, 3, 0), np.delete(x1, 3, 0))
    assert not np.array_equal(x0[3], x1[3])
