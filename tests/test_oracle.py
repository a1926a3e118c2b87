"""Pins for the FP64 oracle (CPU only).

The pages print no worked values, so the oracle is pinned to things other than
itself: hand-worked special cases, closed forms, invariants of the recurrence,
agreement of two independent formulations (token recurrence vs chunked WY
form), and brute force on tiny inputs.  ``test_oracle_mutations.py`` plants
plausible mistakes in the oracle and checks that these pins catch them.
"""

import numpy as np
import pytest

from oracle import kda_ref as ref

RTOL = 1e-10


def _rand_inputs(seed, B, T, Hq, Hv, K, V, N=None, gate=1 / 16, with_h0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, K))
    k = rng.standard_normal((B, T, Hq, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, V))
    g = -np.logaddexp(0, rng.standard_normal((B, T, Hv, K))) * gate
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, Hv))))
    n = B if N is None else N
    h0 = 0.1 * rng.standard_normal((n, Hv, K, V)) if with_h0 else None
    return q, k, v, g, beta, h0


def _close(a, b, rtol=RTOL):
    scale = max(np.max(np.abs(b)), 1e-300)
    return np.max(np.abs(a - b)) / scale <= rtol


# ---------------------------------------------------------------------------
# hand-worked special cases (exact arithmetic, derivations inline)
# ---------------------------------------------------------------------------

def test_scalar_recurrence_hand_worked():
    # K = V = 1, scale = 1.  Each step: decay by e^g, then the delta-rule update
    # S <- (1 - beta k^2) S + beta k v; o = S q.
    # t=1: S0=4, e^g=1/2 -> 2; (1 - 1/2*1)*2 + 1/2*1*2 = 2;        o = 1*2  = 2
    # t=2: e^g=1/4 -> 0.5; (1 - 1/8*4)*0.5 + 1/8*2*8 = 2.25;       o = 3*2.25 = 6.75
    # t=3: e^g=1 -> 2.25; (1 - 1*1)*2.25 + 1*1*(-1) = -1;          o = -2*-1 = 2
    # (decaying after the update instead would give 1.5 at t=1.)
    g = np.log([0.5, 0.25, 1.0]).reshape(1, 3, 1, 1)
    k = np.array([1.0, 2.0, 1.0]).reshape(1, 3, 1, 1)
    beta = np.array([0.5, 0.125, 1.0]).reshape(1, 3, 1)
    v = np.array([2.0, 8.0, -1.0]).reshape(1, 3, 1, 1)
    q = np.array([1.0, 3.0, -2.0]).reshape(1, 3, 1, 1)
    h0 = np.array([4.0]).reshape(1, 1, 1, 1)
    want_o = np.array([2.0, 6.75, 2.0])
    o1, s1 = ref.kda_recurrent(q, k, v, g, beta, 1.0, h0)
    np.testing.assert_allclose(o1.reshape(-1), want_o, rtol=1e-14)
    np.testing.assert_allclose(s1.reshape(-1), [-1.0], rtol=1e-14)
    for C in (1, 2, 64):
        out = ref.kda_chunked(q, k, v, g, beta, 1.0, h0, chunk_size=C)
        np.testing.assert_allclose(out["o"].reshape(-1), want_o, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(out["final_state"].reshape(-1), [-1.0], rtol=1e-13)


def test_vector_recurrence_hand_worked():
    # K = 2, V = 1, scale = 1; per-channel gates.
    # t=1: S0=[1,2], e^g=[1/2,1] -> [0.5,2]; k=[0.6,0.8], k.S=1.9, beta=1, v=5
    #      S1 = [0.5,2] + [0.6,0.8]*(5-1.9) = [2.36, 4.48];  q=[1,1] -> o=6.84
    # t=2: e^g=[1,1/4] -> [2.36,1.12]; k=[1,0], k.S=2.36, beta=1/2, v=1
    #      S2 = [2.36,1.12] + 1/2*[1,0]*(1-2.36) = [1.68, 1.12];  q=[0,2] -> o=2.24
    g = np.log(np.array([[0.5, 1.0], [1.0, 0.25]])).reshape(1, 2, 1, 2)
    k = np.array([[0.6, 0.8], [1.0, 0.0]]).reshape(1, 2, 1, 2)
    q = np.array([[1.0, 1.0], [0.0, 2.0]]).reshape(1, 2, 1, 2)
    v = np.array([5.0, 1.0]).reshape(1, 2, 1, 1)
    beta = np.array([1.0, 0.5]).reshape(1, 2, 1)
    h0 = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    o1, s1 = ref.kda_recurrent(q, k, v, g, beta, 1.0, h0)
    np.testing.assert_allclose(o1.reshape(-1), [6.84, 2.24], rtol=1e-13)
    np.testing.assert_allclose(s1.reshape(-1), [1.68, 1.12], rtol=1e-13)
    out = ref.kda_chunked(q, k, v, g, beta, 1.0, h0, chunk_size=64)
    np.testing.assert_allclose(out["o"].reshape(-1), [6.84, 2.24], rtol=1e-13)
    np.testing.assert_allclose(out["final_state"].reshape(-1), [1.68, 1.12], rtol=1e-13)
    # the intra-chunk pieces of this 2-row chunk, by hand:
    # G = [[ln1/2, 0], [ln1/2, ln1/4]];  Akk[1,0] = beta_1 * sum_c k1 k0 e^{G1-G0}
    #   = 1/2 * (1*0.6*1 + 0*0.8*1/4) = 0.3;  Akk_inv = [[1,0],[-0.3,1]]
    # Aqk[1,0] = sum_c q1 k0 e^{G1-G0} = 0*0.6*1 + 2*0.8*1/4 = 0.4;  Aqk[1,1] = q1.k1 = 0
    # Aqk[0,0] = q0.k0 = 1.4
    np.testing.assert_allclose(out["Akk"][0, :, 0, :2], [[0, 0], [0.3, 0]], atol=1e-15)
    np.testing.assert_allclose(out["Akk_inv"][0, :, 0, :2], [[1, 0], [-0.3, 1]], atol=1e-15)
    np.testing.assert_allclose(out["Aqk"][0, :, 0, :2], [[1.4, 0], [0.4, 0]], atol=1e-15)


# ---------------------------------------------------------------------------
# the two formulations agree (chunk sizes, tails, varlen, GVA)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("T", [1, 37, 130])
def test_chunked_equals_recurrent(C, T):
    q, k, v, g, beta, h0 = _rand_inputs(10 + T, B=2, T=T, Hq=2, Hv=2, K=16, V=8)
    o1, s1 = ref.kda_recurrent(q, k, v, g, beta, 0.25, h0)
    out = ref.kda_chunked(q, k, v, g, beta, 0.25, h0, chunk_size=C)
    assert _close(out["o"], o1)
    assert _close(out["final_state"], s1)


def test_chunked_equals_recurrent_varlen_gva():
    lens = [1, 63, 64, 65, 130, 0, 7]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = _rand_inputs(7, B=1, T=T, Hq=2, Hv=4, K=16, V=8, N=len(lens))
    o1, s1 = ref.kda_recurrent(q, k, v, g, beta, 0.3, h0, cu_seqlens=cu)
    out = ref.kda_chunked(q, k, v, g, beta, 0.3, h0, cu_seqlens=cu, chunk_size=64)
    assert _close(out["o"], o1)
    assert _close(out["final_state"], s1)
    # empty sequence: final = initial
    np.testing.assert_array_equal(out["final_state"][5], h0[5])


def test_chunk_size_invariance():
    q, k, v, g, beta, h0 = _rand_inputs(3, B=1, T=200, Hq=1, Hv=1, K=32, V=16)
    outs = [ref.kda_chunked(q, k, v, g, beta, 0.2, h0, chunk_size=C) for C in (8, 32, 64)]
    for o in outs[1:]:
        assert _close(o["o"], outs[0]["o"])
        assert _close(o["final_state"], outs[0]["final_state"])


# ---------------------------------------------------------------------------
# intra-chunk pieces against definitions that do not reuse the oracle's code
# ---------------------------------------------------------------------------

def _chunk(seed=5, L=64, K=32, V=16):
    q, k, v, g, beta, _ = _rand_inputs(seed, B=1, T=L, Hq=1, Hv=1, K=K, V=V, with_h0=False)
    return q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0]


def test_inverse_is_inverse():
    q, k, v, g, beta = _chunk()
    out = ref.kda_chunked(q[None, :, None], k[None, :, None], v[None, :, None],
                          g[None, :, None], beta[None, :, None], 0.2, chunk_size=64)
    A = out["Akk"][0, :, 0]
    X = out["Akk_inv"][0, :, 0]
    I = np.eye(64)
    assert np.max(np.abs((I + A) @ X - I)) < 1e-10
    assert np.max(np.abs(X @ (I + A) - I)) < 1e-10
    assert np.all(np.triu(X, 1) == 0) and np.all(np.diag(X) == 1)


def test_intra_matrices_brute_force_products_of_gates():
    # decay between rows i <= r is the product of the per-step gates i+1..r
    # (no cumsum, no exp of a difference): pins the inclusive cumsum, the
    # diagonal, the masks, beta on the row side and the scale.
    L, K = 9, 5
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((L, K)), rng.standard_normal((L, K))
    g = -rng.random((L, K))
    beta = rng.random(L)
    scale = 0.37
    Aqk_bf = np.zeros((L, L))
    Akk_bf = np.zeros((L, L))
    for r in range(L):
        for i in range(r + 1):
            for c in range(K):
                d = 1.0
                for j in range(i + 1, r + 1):
                    d *= np.exp(g[j, c])
                Aqk_bf[r, i] += scale * q[r, c] * k[i, c] * d
                if i < r:
                    Akk_bf[r, i] += beta[r] * k[r, c] * k[i, c] * d
    G = ref.chunk_local_cumsum(g)
    Aqk, Akk = ref.intra_chunk_matrices(q, k, G, beta, scale)
    np.testing.assert_allclose(Aqk, Aqk_bf, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Akk, Akk_bf, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(G[3], g[:4].sum(0), rtol=1e-14)


def test_w_u_solve_the_triangular_systems():
    # W and U solve (I + Akk) W = diag(beta)(k * e^G), (I + Akk) U = diag(beta) v,
    # and Delta = U - W S0 solves (I + Akk) Delta = diag(beta)(v - (k*e^G) S0).
    q, k, v, g, beta = _chunk(seed=8)
    G = np.cumsum(g, axis=0)
    _, Akk = ref.intra_chunk_matrices(q, k, G, beta, 0.2)
    X = ref.invert_unit_lower(Akk)
    W, U = ref.recompute_w_u(X, k, v, G, beta)
    I = np.eye(64)
    kg = k * np.exp(G)
    np.testing.assert_allclose((I + Akk) @ W, beta[:, None] * kg, atol=1e-12)
    np.testing.assert_allclose((I + Akk) @ U, beta[:, None] * v, atol=1e-12)
    S0 = np.random.default_rng(2).standard_normal((32, 16))
    D = U - W @ S0
    np.testing.assert_allclose((I + Akk) @ D, beta[:, None] * (v - kg @ S0), atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and invariants of the recurrence
# ---------------------------------------------------------------------------

def test_beta_zero_is_pure_gated_decay():
    q, k, v, g, beta, h0 = _rand_inputs(21, B=1, T=150, Hq=2, Hv=2, K=16, V=8)
    beta = np.zeros_like(beta)
    scale = 0.25
    cum = np.cumsum(g[0], axis=0)                                 # [T, H, K]
    o_want = scale * np.einsum("thk,hkv->thv", q[0] * np.exp(cum), h0[0])
    s_want = np.exp(cum[-1])[:, :, None] * h0[0]
    for fn in ("rec", "chunk"):
        if fn == "rec":
            o, s = ref.kda_recurrent(q, k, v, g, beta, scale, h0)
        else:
            out = ref.kda_chunked(q, k, v, g, beta, scale, h0, chunk_size=64)
            o, s = out["o"], out["final_state"]
        assert _close(o[0], o_want, 1e-12)
        assert _close(s[0], s_want, 1e-12)


def test_orthonormal_keys_store_and_retrieve():
    # g = 0, beta = 1, orthonormal keys, S0 = 0: S_T = sum_t k_t v_t^T and
    # querying with k_j / scale returns v_j for every j <= t.
    K, V, T = 16, 8, 12
    rng = np.random.default_rng(4)
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:, :T].T                                          # [T, K] orthonormal rows
    vals = rng.standard_normal((T, V))
    scale = 0.5
    j_of_t = [rng.integers(0, t + 1) for t in range(T)]
    q = np.stack([keys[j] / scale for j in j_of_t])
    args = (q[None, :, None], keys[None, :, None], vals[None, :, None],
            np.zeros((1, T, 1, K)), np.ones((1, T, 1)), scale)
    o, s = ref.kda_recurrent(*args)
    out = ref.kda_chunked(*args, chunk_size=8)
    for oo, ss in ((o, s), (out["o"], out["final_state"])):
        np.testing.assert_allclose(ss[0, 0], keys.T @ vals, atol=1e-12)
        np.testing.assert_allclose(oo[0, :, 0], vals[j_of_t], atol=1e-12)


def test_rewrite_same_key_overwrites_value():
    # beta = 1, unit key written twice: the delta rule replaces the old value.
    K, V = 8, 4
    rng = np.random.default_rng(9)
    key = rng.standard_normal(K)
    key /= np.linalg.norm(key)
    v1, v2 = rng.standard_normal(V), rng.standard_normal(V)
    args = (np.stack([key, key])[None, :, None], np.stack([key, key])[None, :, None],
            np.stack([v1, v2])[None, :, None], np.zeros((1, 2, 1, K)), np.ones((1, 2, 1)), 1.0)
    for o, s in (ref.kda_recurrent(*args),
                 (lambda d: (d["o"], d["final_state"]))(ref.kda_chunked(*args, chunk_size=2))):
        np.testing.assert_allclose(o[0, 0, 0], v1, atol=1e-12)
        np.testing.assert_allclose(o[0, 1, 0], v2, atol=1e-12)
        np.testing.assert_allclose(s[0, 0], np.outer(key, v2), atol=1e-12)


def test_linearity_in_values_and_initial_state():
    q, k, v, g, beta, h0 = _rand_inputs(31, B=1, T=70, Hq=1, Hv=1, K=16, V=8)
    f = lambda vv, hh: ref.kda_chunked(q, k, vv, g, beta, 0.3, hh, chunk_size=16)
    a, b = f(v, h0), f(v, None)
    c = f(np.zeros_like(v), h0)
    # affine in S0: o(v, S0) = o(v, 0) + o(0, S0)
    assert _close(a["o"], b["o"] + c["o"], 1e-12)
    assert _close(a["final_state"], b["final_state"] + c["final_state"], 1e-12)
    # linear in v when S0 = 0
    d = f(2.5 * v, None)
    assert _close(d["o"], 2.5 * b["o"], 1e-12)


def test_varlen_equals_separate_runs():
    lens = [5, 64, 100, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = _rand_inputs(41, B=1, T=sum(lens), Hq=1, Hv=2, K=16, V=8, N=len(lens))
    packed = ref.kda_chunked(q, k, v, g, beta, 0.3, h0, cu_seqlens=cu, chunk_size=64)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        one = ref.kda_chunked(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e],
                              0.3, h0[n:n + 1], chunk_size=64)
        assert _close(packed["o"][:, s:e], one["o"], 1e-13)
        assert _close(packed["final_state"][n], one["final_state"][0], 1e-13)


def test_gva_equals_mha_with_repeated_qk():
    q, k, v, g, beta, h0 = _rand_inputs(51, B=1, T=80, Hq=2, Hv=6, K=16, V=8)
    gva = ref.kda_chunked(q, k, v, g, beta, 0.3, h0, chunk_size=32)
    mha = ref.kda_chunked(np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2), v, g, beta,
                          0.3, h0, chunk_size=32)
    for key in ("o", "final_state", "Akk_inv", "W", "U", "Aqk"):
        assert _close(gva[key], mha[key], 1e-13)


def test_continuation_across_calls():
    q, k, v, g, beta, h0 = _rand_inputs(61, B=1, T=150, Hq=1, Hv=2, K=16, V=8)
    T1 = 70
    full = ref.kda_chunked(q, k, v, g, beta, 0.3, h0, chunk_size=64)
    first = ref.kda_chunked(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], 0.3, h0)
    second = ref.kda_chunked(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], 0.3,
                             first["final_state"])
    assert _close(full["o"][:, T1:], second["o"], 1e-12)
    assert _close(full["final_state"], second["final_state"], 1e-12)


def test_heads_subset_matches_full():
    q, k, v, g, beta, h0 = _rand_inputs(71, B=1, T=66, Hq=2, Hv=4, K=16, V=8)
    full = ref.kda_chunked(q, k, v, g, beta, 0.3, h0)
    part = ref.kda_chunked(q, k, v, g, beta, 0.3, h0, heads=[1, 3])
    for key in ("o", "W", "Akk_inv"):
        np.testing.assert_array_equal(part[key][:, :, [1, 3]], full[key][:, :, [1, 3]])
    o1, s1 = ref.kda_recurrent(q, k, v, g, beta, 0.3, h0, heads=[2])
    assert _close(o1[:, :, 2], full["o"][:, :, 2])


# ---------------------------------------------------------------------------
# varlen chunk metadata
# ---------------------------------------------------------------------------

def _brute_force_pairs(lens, C):
    # walk the tokens: token t of sequence n lies in chunk (t - bos) // C;
    # the distinct (n, chunk) pairs in token order are the chunk list.
    seen = []
    for n, ln in enumerate(lens):
        for t in range(ln):
            p = (n, t // C)
            if not seen or seen[-1] != p:
                seen.append(p)
    return seen


@pytest.mark.parametrize("lens", [[1], [64], [65], [1, 63, 64, 65, 0, 129, 3], [0, 0], []])
@pytest.mark.parametrize("C", [16, 64])
def test_chunk_indices_brute_force(lens, C):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx, off = ref.prepare_chunk_indices(cu, C)
    want = _brute_force_pairs(lens, C)
    assert idx.dtype == np.int32 and idx.shape == (len(want), 2)
    assert [tuple(x) for x in idx.tolist()] == want
    assert off[0] == 0 and len(off) == len(lens) + 1
    for n in range(len(lens)):
        assert off[n + 1] - off[n] == sum(1 for p in want if p[0] == n)
    assert len(want) <= ref.num_chunks_bound(int(cu[-1]), len(lens), C)


@pytest.mark.parametrize("bad", [None, 0, -64, True, 1.5])
def test_chunk_indices_reject_bad_chunk_size(bad):
    with pytest.raises(ValueError):
        ref.prepare_chunk_indices(np.array([0, 4], np.int32), bad)


def test_chunk_indices_reject_unsorted():
    with pytest.raises(ValueError):
        ref.prepare_chunk_indices(np.array([0, 10, 4], np.int32), 64)


def test_chunk_indices_empty():
    idx, off = ref.prepare_chunk_indices(np.array([0], np.int32), 64)
    assert idx.shape == (0, 2) and off.tolist() == [0]


# ---------------------------------------------------------------------------
# the optional gated query QG = q * e^G (cuLA PR #131, Summary: optional QG)
# ---------------------------------------------------------------------------

def test_gated_query_closed_form_constant_gates():
    # Gates constant in time (per value head and channel): row r of a chunk
    # (counting from 0 at the chunk start, the count restarting at every chunk
    # and sequence) carries q * exp((r + 1) * g).  Value head hv reads the q
    # of q/k head hv // (Hv // Hq).  Packed varlen with ragged sequences.
    rng = np.random.default_rng(91)
    lens = [70, 5, 130]
    T, Hq, Hv, K, V = sum(lens), 2, 4, 8, 4
    cu = np.concatenate([[0], np.cumsum(lens)])
    q = rng.standard_normal((1, T, Hq, K))
    k = rng.standard_normal((1, T, Hq, K)) * 0.1
    v = rng.standard_normal((1, T, Hv, V))
    gc = -rng.uniform(0.01, 0.2, size=(Hv, K))
    g = np.broadcast_to(gc, (1, T, Hv, K)).copy()
    beta = np.full((1, T, Hv), 0.5)
    out = ref.kda_chunked(q, k, v, g, beta, 0.3, None, cu, chunk_size=64)
    want = np.zeros((1, T, Hv, K))
    for bos, eos in zip(cu[:-1], cu[1:]):
        for t in range(bos, eos):
            r = (t - bos) % 64
            for hv in range(Hv):
                want[0, t, hv] = q[0, t, hv // (Hv // Hq)] * np.exp((r + 1) * gc[hv])
    assert _close(out["QG"], want)


def test_gated_query_brute_force_products():
    # Random gates: QG[t] = q[t] * prod_{j = chunk start .. t} exp(g_j), a
    # running product of per-token factors (no cumsum of logs).
    q, k, v, g, beta, _ = _rand_inputs(92, B=2, T=150, Hq=1, Hv=2, K=4, V=3, with_h0=False)
    out = ref.kda_chunked(q, k, v, g, beta, 0.5, None, None, chunk_size=64)
    want = np.zeros_like(out["QG"])
    for b in range(2):
        for hv in range(2):
            prod = np.ones(4)
            for t in range(150):
                if t % 64 == 0:
                    prod = np.ones(4)
                prod = prod * np.exp(g[b, t, hv])
                want[b, t, hv] = q[b, t, 0] * prod
    assert _close(out["QG"], want)
