"""Pins for the CPU oracle (runs without a GPU).

The oracle is checked against things other than itself: hand-worked fixtures
from the paper's equations (tests/golden), library routines on the special
cases where the method reduces to one (stable argsort; dense matmul and
scipy's logistic sigmoid for the all-ones mask), invariants the equations
imply (permutation, prefix identity, complement linearity, token and group
permutation), and brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from group_masked_gemm_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf(x):
    """float array (exactly representable) -> bf16 bits."""
    b = syn.bf16_bits(np.asarray(x, np.float32))
    assert np.array_equal(syn.bf16_to_f32(b), np.asarray(x, np.float32))
    return b


def _closed(expr):
    return eval(expr, {"__builtins__": {}}, {"exp": math.exp})


def _f64(bits):
    return syn.bf16_to_f32(bits).astype(np.float64)


def _swiglu_dense(inp):
    """Dense SwiGLU FFN with library routines: numpy matmul + scipy expit."""
    X, Wg, Wu, Wd = (_f64(a) for a in (inp.X, inp.Wg, inp.Wu, inp.Wd))
    a = X @ Wg.T
    b = X @ Wu.T
    h = a * expit(a) * b
    return h, h @ Wd.T


def _expand(mask, G):
    return np.repeat(mask.astype(bool), G, axis=1)


# --- reorder (Eq. 7) ----------------------------------------------------------

def test_reorder_golden_eq7():
    g = _load("reorder_eq7_example.json")
    mask = np.array(g["mask_rows"], np.uint8)
    perm, counts = oracle.reorder(mask)
    assert perm.tolist() == g["perm"]
    assert counts.tolist() == g["counts"]


@pytest.mark.parametrize("T,ng,keep,seed", [
    (1, 1, 0.5, 0), (7, 3, 0.5, 1), (64, 8, 0.5, 2), (300, 28, 0.3, 3),
    (1000, 112, 0.5, 4), (257, 5, 0.9, 5), (129, 224, 0.1, 6)])
def test_reorder_matches_stable_argsort(T, ng, keep, seed):
    mask = syn.random_mask(T, ng, keep, seed)
    perm, counts = oracle.reorder(mask)
    for g in range(ng):
        ref = np.argsort(-(mask[:, g] != 0).astype(np.int64), kind="stable")
        assert np.array_equal(perm[g], ref)
    assert np.array_equal(counts, (mask != 0).sum(0))


@pytest.mark.parametrize("BM", [64, 128])
def test_reorder_invariants(BM):
    mask = syn.random_mask(1500, 37, 0.45, 11)
    mask[3, :] = 255                      # any nonzero byte is active
    mask[:, 0] = 0                        # an empty group
    mask[:, 1] = 1                        # a full group
    perm, counts = oracle.reorder(mask)
    T, ng = mask.shape
    for g in range(ng):
        p, c = perm[g], counts[g]
        assert sorted(p.tolist()) == list(range(T))            # a permutation
        act = mask[p, g] != 0
        assert act[:c].all() and not act[c:].any()             # prefix identity
        assert np.all(np.diff(p[:c]) > 0) and np.all(np.diff(p[c:]) > 0)
        # Sec. 3.3: at most one partially active BM-row tile per group
        tiles = [act[i:i + BM] for i in range(0, T, BM)]
        partial = [t for t in tiles if t.any() and not t.all()]
        assert len(partial) <= 1
    assert counts[0] == 0 and counts[1] == T


def test_reorder_brute_force_tiny():
    rng = np.random.default_rng(99)
    for _ in range(50):
        T = int(rng.integers(1, 12))
        ng = int(rng.integers(1, 5))
        mask = (rng.random((T, ng)) < 0.5).astype(np.uint8)
        perm, counts = oracle.reorder(mask)
        for g in range(ng):
            act = [t for t in range(T) if mask[t, g]]
            ina = [t for t in range(T) if not mask[t, g]]
            assert perm[g].tolist() == act + ina
            assert counts[g] == len(act)


# --- closed-form fixtures ------------------------------------------------------

def test_ffn_golden_closed_form():
    g = _load("ffn_closed_form.json")
    X, Wg, Wu, Wd = (_bf(g[k]) for k in ("X", "Wg", "Wu", "Wd"))
    mask = np.array(g["mask"], np.uint8)
    H = oracle.gate_up(X, Wg, Wu, mask, g["G"])
    Y = oracle.ffn(X, Wg, Wu, Wd, mask, g["G"])
    Hx = np.array([[_closed(e) for e in r] for r in g["H"]])
    Yx = np.array([[_closed(e) for e in r] for r in g["Y"]])
    np.testing.assert_allclose(H, Hx, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(Y, Yx, rtol=1e-14, atol=1e-15)


def test_proj_golden_closed_form():
    g = _load("proj_closed_form.json")
    mn, k = g["proj_mn"], g["proj_k"]
    Y = oracle.proj_mn(_bf(mn["X"]), _bf(mn["W"]), np.array(mn["mask"], np.uint8), mn["G"])
    assert np.array_equal(Y, np.array(mn["Y"], np.float64))
    Y = oracle.proj_k(_bf(k["A"]), _bf(k["W"]), np.array(k["mask"], np.uint8), k["G"])
    assert np.array_equal(Y, np.array(k["Y"], np.float64))


# --- special cases that reduce to library routines -------------------------------

@pytest.fixture(scope="module")
def tiny():
    return syn.tiny_ffn()


def test_all_ones_is_dense_swiglu(tiny):
    ones = syn.with_mask(tiny, np.ones_like(tiny.mask))
    h_ref, y_ref = _swiglu_dense(ones)
    H = oracle.gate_up(ones.X, ones.Wg, ones.Wu, ones.mask, ones.G)
    Y = oracle.ffn(ones.X, ones.Wg, ones.Wu, ones.Wd, ones.mask, ones.G)
    np.testing.assert_allclose(H, h_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Y, y_ref, rtol=1e-10, atol=1e-12)


def test_all_zeros_is_zero(tiny):
    z = np.zeros_like(tiny.mask)
    assert not oracle.gate_up(tiny.X, tiny.Wg, tiny.Wu, z, tiny.G).any()
    assert not oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, z, tiny.G).any()
    assert not oracle.proj_mn(tiny.X, tiny.Wg, z, tiny.G).any()
    A = tiny.X[:, :0]
    A = syn.bf16_bits(np.ones((tiny.T, tiny.F), np.float32))
    assert not oracle.proj_k(A, tiny.Wd, z, tiny.G).any()


def test_masked_gate_up_equals_masked_dense(tiny):
    h_ref, _ = _swiglu_dense(tiny)
    h_ref = np.where(_expand(tiny.mask, tiny.G), h_ref, 0.0)
    H = oracle.gate_up(tiny.X, tiny.Wg, tiny.Wu, tiny.mask, tiny.G)
    np.testing.assert_allclose(H, h_ref, rtol=1e-10, atol=1e-12)


def test_proj_mn_equals_masked_matmul():
    rng = np.random.default_rng(5)
    T, K, N, G = 33, 96, 160, 32
    X = syn.bf16_bits(rng.standard_normal((T, K), dtype=np.float32))
    W = syn.bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    mask = (rng.random((T, N // G)) < 0.5).astype(np.uint8)
    ref = np.where(_expand(mask, G), _f64(X) @ _f64(W).T, 0.0)
    np.testing.assert_allclose(oracle.proj_mn(X, W, mask, G), ref, rtol=1e-10, atol=1e-12)


def test_proj_k_equals_matmul_of_masked_A():
    rng = np.random.default_rng(6)
    T, K, N, G = 29, 256, 72, 64
    A = syn.bf16_bits(rng.standard_normal((T, K), dtype=np.float32))
    W = syn.bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    mask = (rng.random((T, K // G)) < 0.5).astype(np.uint8)
    ref = np.where(_expand(mask, G), _f64(A), 0.0) @ _f64(W).T
    np.testing.assert_allclose(oracle.proj_k(A, W, mask, G), ref, rtol=1e-10, atol=1e-12)
    ones = np.ones_like(mask)
    np.testing.assert_allclose(oracle.proj_k(A, W, ones, G), _f64(A) @ _f64(W).T,
                               rtol=1e-10, atol=1e-12)


def test_single_group_mask_is_dense_slice(tiny):
    g = 3
    m = np.zeros_like(tiny.mask)
    m[:, g] = 1
    G = tiny.G
    X, Wg, Wu, Wd = (_f64(a) for a in (tiny.X, tiny.Wg, tiny.Wu, tiny.Wd))
    sl = slice(g * G, (g + 1) * G)
    a = X @ Wg[sl].T
    h = a * expit(a) * (X @ Wu[sl].T)
    y_ref = h @ Wd[:, sl].T
    Y = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, m, G)
    np.testing.assert_allclose(Y, y_ref, rtol=1e-10, atol=1e-12)


def test_whole_width_group_is_token_mask_times_dense(tiny):
    """N_G = 1 (App. B: M-axis depth is the one-group case of GEMM-MN/GEMM-K):
    every token either gets the whole dense row or zero."""
    rng = np.random.default_rng(5)
    T = tiny.T
    m = (rng.random((T, 1)) < 0.5).astype(np.uint8)
    X, Wg, Wu, Wd = (_f64(a) for a in (tiny.X, tiny.Wg, tiny.Wu, tiny.Wd))
    keep = m[:, :1].astype(np.float64)
    np.testing.assert_allclose(oracle.proj_mn(tiny.X, tiny.Wg, m, tiny.F), keep * (X @ Wg.T),
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(oracle.proj_k(tiny.X, tiny.Wg, m, tiny.D), keep * (X @ Wg.T),
                               rtol=1e-10, atol=1e-12)
    a = X @ Wg.T
    y = keep * ((a * expit(a) * (X @ Wu.T)) @ Wd.T)
    np.testing.assert_allclose(oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, m, tiny.F), y,
                               rtol=1e-10, atol=1e-12)


def test_router_golden_eq4_5():
    with open(os.path.join(GOLDEN, "router_eq4_5_example.json")) as f:
        gold = json.load(f)
    X, W1, W2 = (syn.bf16_bits(np.array(gold[k], np.float32)) for k in ("X", "W1", "W2"))
    logits, mask = oracle.router(X, W1, W2)
    np.testing.assert_array_equal(logits, np.array(gold["logits"], np.float64))
    np.testing.assert_array_equal(mask, np.array(gold["mask"], np.uint8))


def _router_inputs(seed, T=96, D=192, r=16, ng=12):
    rng = np.random.default_rng(seed)
    X = syn.bf16_bits(rng.standard_normal((T, D), dtype=np.float32))
    W1 = syn.bf16_bits(rng.standard_normal((r, D), dtype=np.float32) * np.float32(D ** -0.5))
    W2 = syn.bf16_bits(rng.standard_normal((2 * ng, r), dtype=np.float32) * np.float32(r ** -0.5))
    return X, W1, W2


def test_router_class_swap_complements_mask():
    """Swapping the two class rows of every group exchanges R0 and R1, so the
    mask flips everywhere except at exact ties (which stay active)."""
    X, W1, W2 = _router_inputs(21)
    logits, mask = oracle.router(X, W1, W2)
    W2s = W2.reshape(-1, 2, W2.shape[1])[:, ::-1, :].reshape(W2.shape).copy()
    logits_s, mask_s = oracle.router(X, W1, W2s)
    np.testing.assert_array_equal(logits_s.reshape(len(X), -1, 2), logits.reshape(len(X), -1, 2)[:, :, ::-1])
    tie = logits[:, 0::2].astype(np.float32) == logits[:, 1::2].astype(np.float32)
    np.testing.assert_array_equal(mask_s[~tie], 1 - mask[~tie])
    assert 0.2 < mask.mean() < 0.8   # random router weights keep about half


def test_router_scale_invariance_and_ties():
    """Doubling X (exact in bf16) doubles every logit and keeps every decision;
    identical class rows give exact ties, which execute (class 0)."""
    X, W1, W2 = _router_inputs(22)
    logits, mask = oracle.router(X, W1, W2)
    X2 = syn.bf16_bits(2.0 * syn.bf16_to_f32(X))
    logits2, mask2 = oracle.router(X2, W1, W2)
    np.testing.assert_array_equal(logits2, 2.0 * logits)
    np.testing.assert_array_equal(mask2, mask)
    W2t = W2.copy()
    W2t[1::2] = W2t[0::2]
    _, mask_t = oracle.router(X, W1, W2t)
    assert mask_t.all()


def test_router_tokens_are_independent():
    X, W1, W2 = _router_inputs(23)
    order = np.random.default_rng(1).permutation(len(X))
    logits, mask = oracle.router(X, W1, W2)
    logits_p, mask_p = oracle.router(X[order].copy(), W1, W2)
    np.testing.assert_array_equal(logits_p, logits[order])
    np.testing.assert_array_equal(mask_p, mask[order])


def test_attn_decode_golden():
    with open(os.path.join(GOLDEN, "attn_decode_example.json")) as f:
        gold = json.load(f)
    Q, K, V = (syn.bf16_bits(np.array(gold[k], np.float32)) for k in ("Q", "K", "V"))
    O = oracle.attn_decode(Q, K, V, np.array(gold["lens"], np.int32), np.array(gold["mask"], np.uint8))
    np.testing.assert_allclose(O, np.array(gold["O"], np.float64), rtol=1e-12, atol=1e-15)


def _attn_inputs(seed, B=3, Hq=8, Hk=2, d=64, L_max=50):
    rng = np.random.default_rng(seed)
    Q = syn.bf16_bits(rng.standard_normal((B, Hq, d), dtype=np.float32))
    K = syn.bf16_bits(rng.standard_normal((B, Hk, L_max, d), dtype=np.float32))
    V = syn.bf16_bits(rng.standard_normal((B, Hk, L_max, d), dtype=np.float32))
    lens = rng.integers(1, L_max + 1, size=B).astype(np.int32)
    return Q, K, V, lens


def test_attn_decode_key_permutation_and_tail():
    """Softmax attention is invariant to permuting the cached (key, value)
    pairs, and nothing past lens[b] is read."""
    Q, K, V, lens = _attn_inputs(31)
    mask = np.ones((Q.shape[0], K.shape[1]), np.uint8)
    O = oracle.attn_decode(Q, K, V, lens, mask)
    K2, V2 = K.copy(), V.copy()
    rng = np.random.default_rng(2)
    for b, L in enumerate(lens):
        p = rng.permutation(L)
        K2[b, :, :L] = K[b, :, p].transpose(1, 0, 2)
        V2[b, :, :L] = V[b, :, p].transpose(1, 0, 2)
        K2[b, :, L:] = 0x7F80  # +inf bit patterns past the end
        V2[b, :, L:] = 0x7F80
    np.testing.assert_allclose(oracle.attn_decode(Q, K2, V2, lens, mask), O, rtol=1e-12, atol=1e-13)


def test_attn_decode_equal_keys_average_and_groups():
    """Equal keys give uniform weights (the mean of the value rows); query
    heads of one GQA group share its KV head; an inactive group is zero."""
    Q, K, V, lens = _attn_inputs(32)
    K[:] = K[:, :, :1, :]
    mask = np.ones((Q.shape[0], K.shape[1]), np.uint8)
    O = oracle.attn_decode(Q, K, V, lens, mask)
    Vf = syn.bf16_to_f32(V).astype(np.float64)
    qpk = Q.shape[1] // K.shape[1]
    for b, L in enumerate(lens):
        for h in range(Q.shape[1]):
            np.testing.assert_allclose(O[b, h], Vf[b, h // qpk, :L].mean(0), rtol=1e-10, atol=1e-12)
    Q2 = Q.copy()
    Q2[:, 1] = Q2[:, 0]  # heads 0 and 1 share KV head 0
    mask[1, 1] = 0
    O2 = oracle.attn_decode(Q2, K, V, lens, mask)
    np.testing.assert_array_equal(O2[:, 0], O2[:, 1])
    assert (O2[1, qpk:2 * qpk] == 0).all()


def test_attn_prefill_golden():
    with open(os.path.join(GOLDEN, "attn_prefill_example.json")) as f:
        gold = json.load(f)
    Q, K, V = (syn.bf16_bits(np.array(gold[k], np.float32)) for k in ("Q", "K", "V"))
    mask = np.array(gold["mask"], np.uint8)
    np.testing.assert_allclose(oracle.attn_prefill(Q, K, V, mask), np.array(gold["O_causal"], np.float64),
                               rtol=1e-12, atol=1e-15)
    ones = np.ones_like(mask)
    np.testing.assert_allclose(oracle.attn_prefill(Q, K, V, ones)[0, 2, 0],
                               gold["O_all_active_causal_t2"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.attn_prefill(Q, K, V, ones, causal=False)[0, 0, 0],
                               gold["O_all_active_noncausal_t0"], rtol=1e-12, atol=1e-15)


def test_attn_prefill_causal_is_prefix_attention():
    """Causal output at position t equals full attention over keys 0..t, and
    matches the decode formulation (one query over a cache of t+1 keys)."""
    rng = np.random.default_rng(41)
    B, T, Hq, Hk, d = 2, 20, 4, 2, 32
    Q = syn.bf16_bits(rng.standard_normal((B, T, Hq, d), dtype=np.float32))
    K = syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32))
    V = syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32))
    mask = (rng.random((B, T, Hk)) < 0.6).astype(np.uint8)
    O = oracle.attn_prefill(Q, K, V, mask)
    for t in (0, 7, 19):
        Ot = oracle.attn_prefill(Q[:, :t + 1].copy(), K[:, :, :t + 1].copy(), V[:, :, :t + 1].copy(),
                                 mask[:, :t + 1].copy(), causal=False)
        np.testing.assert_allclose(O[:, t], Ot[:, t], rtol=1e-12, atol=1e-14)
        Od = oracle.attn_decode(Q[:, t].copy(), K, V, np.full(B, t + 1, np.int32), mask[:, t].copy())
        np.testing.assert_allclose(O[:, t], Od, rtol=1e-12, atol=1e-14)
    qpk = Hq // Hk
    for b in range(B):
        for t in range(T):
            for g in range(Hk):
                if mask[b, t, g] == 0:
                    assert (O[b, t, g * qpk:(g + 1) * qpk] == 0).all()


# --- invariants ---------------------------------------------------------------------

def test_complement_linearity(tiny):
    y1 = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask, tiny.G)
    y2 = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, 1 - tiny.mask, tiny.G)
    y_all = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, np.ones_like(tiny.mask), tiny.G)
    np.testing.assert_allclose(y1 + y2, y_all, rtol=1e-9, atol=1e-12)


def test_token_permutation_commutes(tiny):
    p = np.random.default_rng(7).permutation(tiny.T)
    y = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask, tiny.G)
    yp = oracle.ffn(tiny.X[p], tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask[p], tiny.G)
    np.testing.assert_array_equal(yp, y[p])


def test_group_permutation_invariance(tiny):
    G, ng = tiny.G, tiny.n_groups
    q = np.random.default_rng(8).permutation(ng)
    cols = np.concatenate([np.arange(g * G, (g + 1) * G) for g in q])
    y = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask, G)
    yq = oracle.ffn(tiny.X, tiny.Wg[cols], tiny.Wu[cols], tiny.Wd[:, cols],
                    tiny.mask[:, q], G)
    np.testing.assert_allclose(yq, y, rtol=1e-12, atol=1e-13)


def test_proj_k_ignores_inactive_entries():
    rng = np.random.default_rng(9)
    T, K, N, G = 40, 512, 64, 128
    A = syn.bf16_bits(rng.standard_normal((T, K), dtype=np.float32))
    W = syn.bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    mask = (rng.random((T, K // G)) < 0.5).astype(np.uint8)
    garbage = syn.bf16_bits(rng.standard_normal((T, K), dtype=np.float32) * 1e3)
    A2 = np.where(_expand(mask, G), A, garbage)
    np.testing.assert_array_equal(oracle.proj_k(A, W, mask, G), oracle.proj_k(A2, W, mask, G))


def test_rows_subset_matches_full(tiny):
    rows = np.array([0, 5, 17, 63], np.int32)
    full = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask, tiny.G)
    sub = oracle.ffn(tiny.X, tiny.Wg, tiny.Wu, tiny.Wd, tiny.mask, tiny.G, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    H = oracle.gate_up(tiny.X, tiny.Wg, tiny.Wu, tiny.mask, tiny.G)
    Hs = oracle.gate_up(tiny.X, tiny.Wg, tiny.Wu, tiny.mask, tiny.G, rows=rows)
    np.testing.assert_array_equal(Hs, H[rows])


def test_brute_force_tiny_ffn():
    """Pure-Python per-element sums on a tiny random case."""
    rng = np.random.default_rng(10)
    T, D, F, G = 3, 4, 6, 2
    X = syn.bf16_bits(rng.standard_normal((T, D), dtype=np.float32))
    Wg = syn.bf16_bits(rng.standard_normal((F, D), dtype=np.float32))
    Wu = syn.bf16_bits(rng.standard_normal((F, D), dtype=np.float32))
    Wd = syn.bf16_bits(rng.standard_normal((D, F), dtype=np.float32))
    mask = (rng.random((T, F // G)) < 0.6).astype(np.uint8)
    x, wg, wu, wd = (_f64(a).tolist() for a in (X, Wg, Wu, Wd))
    y = [[0.0] * D for _ in range(T)]
    for t in range(T):
        h = []
        for f in range(F):
            a = sum(x[t][d] * wg[f][d] for d in range(D))
            b = sum(x[t][d] * wu[f][d] for d in range(D))
            h.append(a * float(expit(a)) * b if mask[t][f // G] else 0.0)
        for n in range(D):
            y[t][n] = sum(h[f] * wd[n][f] for f in range(F))
    np.testing.assert_allclose(oracle.ffn(X, Wg, Wu, Wd, mask, G), np.array(y),
                               rtol=1e-12, atol=1e-14)
