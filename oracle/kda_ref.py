"""FP64 CPU oracle for the chunked KDA (Kimi Delta Attention) forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import or run it.  The CUDA library has no CPU fallback; it
fails loudly when its shared object is missing.

What it computes
----------------
KDA is the delta rule with a per-channel (diagonal) forget gate.  For one value
head, with state ``S`` of shape ``[K, V]``, every token ``t`` applies

    S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
    o_t = scale * S_t^T q_t

cuLA REPO_LAYOUT.md lists the KDA operator package (cula/kda/) and the two
kernels of its modular forward that run after the intra-chunk work: the delta-H
state kernel (chunk_delta_h.py) and the output kernel (fwd_o.py).  cuLA PR #131
(Summary) ports the three intra-chunk steps: the intra-chunk matrices, the FP32
inverse of Akk, and the W/U recompute.  None of the pages writes the recurrence
out, so the token recurrence above is the definition this oracle starts from.

Two independent implementations live here:

* ``kda_recurrent`` (O1) -- the token-by-token recurrence, the plain definition.
* ``kda_chunked``   (O2) -- the chunked (WY) form that the named steps compute:
  in-chunk gate cumsum, Aqk / Akk, the inverse of (I + Akk), W / U, then the
  inter-chunk state pass (delta-H) and the output (fwd_o).

Derivation of O2 from O1 (inside one chunk of L rows, state S0 at its start,
G_r = sum_{j<=r} g_j the inclusive in-chunk cumsum):
  with S^_r = Diag(e^{g_r}) S_{r-1} and delta_r = beta_r (v_r - S^_r^T k_r),
  S_r = S^_r + k_r delta_r^T, so
  S_r = Diag(e^{G_r}) S0 + sum_{i<=r} Diag(e^{G_r - G_i}) k_i delta_i^T.
  Substituting into delta_r gives (I + Akk) Delta = diag(beta) V - diag(beta)(K*e^G) S0
  with Akk[r,i] = beta_r sum_c k_r[c] k_i[c] e^{G_r[c]-G_i[c]} (i < r), hence
  Delta = U - W S0 with W = (I+Akk)^{-1} diag(beta)(K*e^G), U = (I+Akk)^{-1} diag(beta) V.
  o_r = scale (q_r*e^{G_r})^T S0 + sum_{i<=r} Aqk[r,i] delta_i with
  Aqk[r,i] = scale sum_c q_r[c] k_i[c] e^{G_r[c]-G_i[c]} (i <= r), and the
  state after the chunk is Diag(e^{G_last}) S0 + (K*e^{G_last-G})^T Delta.

Readings taken where the pages are silent:
  * Akk is stored positive, beta-scaled and strictly lower triangular;
    Akk_inv = (I + Akk)^{-1} includes its unit diagonal and is zero above it.
  * Aqk includes ``scale`` and its diagonal.
  * The cumsum is inclusive and restarts at every chunk and every sequence.
  * Grouped-value heads: g and beta are per value head; value head hv reads
    q/k head hv // (Hv // Hq).
  * A partial tail chunk has L < C rows; rows >= L do not exist.  Entries of
    Aqk / Akk_inv in columns >= L are zero, and the state after a tail chunk
    decays with G[L-1].

Layouts (token-major, as the CUDA path uses):
  q, k [B, T, Hq, K]; v [B, T, Hv, V]; g [B, T, Hv, K]; beta [B, T, Hv];
  initial / final state [N, Hv, K, V] (N = B, or the number of packed
  sequences when ``cu_seqlens`` is given, in which case B must be 1);
  o [B, T, Hv, V]; Aqk, Akk, Akk_inv [B, T, Hv, C] (row t holds row t-t0 of its
  chunk's C x C matrix); W [B, T, Hv, K]; U [B, T, Hv, V]; G [B, T, Hv, K].

Parity pins: every function here is checked in ``tests/test_oracle.py``
against closed forms, invariants and brute force that do not reuse this code.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "sequences",
    "kda_recurrent",
    "chunk_local_cumsum",
    "intra_chunk_matrices",
    "invert_unit_lower",
    "recompute_w_u",
    "chunk_state_output",
    "kda_chunked",
    "gated_query",
    "prepare_lens",
    "prepare_chunk_indices",
]


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def sequences(B, T, cu_seqlens=None):
    """List the sequences as (batch row, first token, end token).

    Fixed length: B sequences of T tokens, one per batch row.  Packed varlen
    (supported per cuLA PR #131, Summary; FLA convention): B == 1 and sequence
    n spans tokens [cu[n], cu[n+1]).
    """
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    if B != 1:
        raise ValueError("packed varlen inputs need B == 1")
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    if len(cu) < 1 or cu[0] != 0 or cu[-1] != T:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    if any(cu[n + 1] < cu[n] for n in range(len(cu) - 1)):
        raise ValueError("cu_seqlens must be non-decreasing")
    return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


# ---------------------------------------------------------------------------
# O1: the token recurrence (the plain definition)
# ---------------------------------------------------------------------------

def kda_recurrent(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None,
                  heads=None):
    """Token-by-token KDA forward in FP64.

    Per token: decay every row c of S by exp(g_t[c]), then apply the delta-rule
    correction S <- S - beta k (k^T S) + beta k v^T, which equals
    (I - beta k k^T) Diag(exp(g)) S_{t-1} + beta k v^T; read out
    o_t = scale S^T q_t.

    ``heads`` restricts the work to a subset of value heads (the other heads'
    outputs are left at zero).  Returns (o [B,T,Hv,V], final [N,Hv,K,V]).
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S0 = _f64(initial_state)
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    grp = Hv // Hq
    hv_list = list(range(Hv)) if heads is None else list(heads)
    hq_list = [hv // grp for hv in hv_list]
    seqs = sequences(B, T, cu_seqlens)
    o = np.zeros((B, T, Hv, V))
    final = np.zeros((len(seqs), Hv, K, V))
    for n, (b, bos, eos) in enumerate(seqs):
        # all selected heads advance together: S has shape [h, K, V]
        S = np.zeros((len(hv_list), K, V)) if S0 is None else S0[n, hv_list].copy()
        for t in range(bos, eos):
            qt = q[b, t, hq_list]            # [h, K]
            kt = k[b, t, hq_list]            # [h, K]
            vt = v[b, t, hv_list]            # [h, V]
            bt = beta[b, t, hv_list]         # [h]
            S = np.exp(g[b, t, hv_list])[:, :, None] * S
            kS = np.einsum("hk,hkv->hv", kt, S)
            S = S + bt[:, None, None] * kt[:, :, None] * (vt - kS)[:, None, :]
            o[b, t, hv_list] = scale * np.einsum("hkv,hk->hv", S, qt)
        final[n, hv_list] = S
    return o, final


# ---------------------------------------------------------------------------
# O2: the chunked form, step by step
# ---------------------------------------------------------------------------

def chunk_local_cumsum(g_chunk):
    """Inclusive cumsum of the log-gates over the rows of one chunk: G[r] = sum_{j<=r} g[j].

    The first step of the intra-chunk work (cuLA PR #131, Summary; its
    Performance section notes the cumsum is a separate, unfused step).
    """
    return np.cumsum(g_chunk, axis=0)


def intra_chunk_matrices(q_c, k_c, G_c, beta_c, scale):
    """Gated, causally masked Aqk and strictly-lower, beta-scaled Akk of one chunk.

    Aqk[r, i] = scale * sum_c q[r,c] k[i,c] exp(G[r,c] - G[i,c])   for i <= r
    Akk[r, i] = beta[r] * sum_c k[r,c] k[i,c] exp(G[r,c] - G[i,c]) for i <  r
    Both zero elsewhere.  The pair exp(G_r - G_i) is formed directly for each
    (r, i, c), never split into exp(G_r) * exp(-G_i).
    Names follow cuLA PR #131 (Summary and Numerical behavior, where Akk is
    the lower-triangular intra-chunk key matrix).
    """
    L = q_c.shape[0]
    lower_incl = np.tril(np.ones((L, L), dtype=bool))
    lower_strict = np.tril(np.ones((L, L), dtype=bool), -1)
    diff = G_c[:, None, :] - G_c[None, :, :]               # [r, i, c]
    decay = np.exp(np.where(lower_incl[:, :, None], diff, -np.inf))
    Aqk = scale * np.einsum("rc,ic,ric->ri", q_c, k_c, decay)
    Akk = beta_c[:, None] * np.einsum("rc,ic,ric->ri", k_c, k_c, decay)
    return np.where(lower_incl, Aqk, 0.0), np.where(lower_strict, Akk, 0.0)


def invert_unit_lower(Akk):
    """(I + Akk)^{-1} by textbook forward substitution, one row at a time.

    Row r of (I + A) X = I reads X[r, :] + sum_{i<r} A[r, i] X[i, :] = e_r.
    Works on a leading batch of matrices.  This is the inverse step of cuLA
    PR #131 (Summary; Numerical behavior, which keeps it in an FP32 workspace),
    done here in FP64.
    """
    A = np.asarray(Akk, dtype=np.float64)
    L = A.shape[-1]
    X = np.zeros_like(A)
    for r in range(L):
        X[..., r, r] = 1.0
        if r:
            X[..., r, :] -= np.einsum("...i,...ij->...j", A[..., r, :r], X[..., :r, :])
    return X


def recompute_w_u(Akk_inv, k_c, v_c, G_c, beta_c):
    """W = Akk_inv (beta * k * exp(G)),  U = Akk_inv (beta * v).

    The W/U recompute step of cuLA PR #131 (Summary).
    """
    W = Akk_inv @ (beta_c[:, None] * k_c * np.exp(G_c))
    U = Akk_inv @ (beta_c[:, None] * v_c)
    return W, U


def chunk_state_output(S0, q_c, k_c, G_c, Aqk, W, U, scale):
    """One chunk of the inter-chunk pass: output rows and the next state.

    Delta = U - W S0
    O     = scale (q * exp(G)) S0 + Aqk Delta
    S1    = Diag(exp(G_last)) S0 + (k * exp(G_last - G))^T Delta
    The delta-H state kernel and the output kernel of cuLA REPO_LAYOUT.md
    (chunk_delta_h.py, fwd_o.py).
    """
    delta = U - W @ S0
    o = scale * (q_c * np.exp(G_c)) @ S0 + Aqk @ delta
    g_last = G_c[-1]
    S1 = np.exp(g_last)[:, None] * S0 + (k_c * np.exp(g_last[None, :] - G_c)).T @ delta
    return o, S1


def gated_query(q_c, G_c):
    """The optional QG output of cuLA PR #131 (Summary: "optional QG"): the
    query of each row gated by its in-chunk cumulative log-gate, q * e^G.
    The pages say no more; it is read per value head, without ``scale``."""
    return q_c * np.exp(G_c)


def kda_chunked(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None,
                chunk_size=64, heads=None):
    """Chunked KDA forward in FP64 (O2), with every intermediate.

    Returns a dict with o [B,T,Hv,V], final_state [N,Hv,K,V], and the
    token-major intermediates Aqk, Akk, Akk_inv [B,T,Hv,C], W [B,T,Hv,K],
    U [B,T,Hv,V], G [B,T,Hv,K] and the gated query QG = q * e^G [B,T,Hv,K]
    (the optional QG output of cuLA PR #131, Summary; per value head, from the
    q/k head it reads).  ``heads`` restricts the work to a subset of value
    heads (the other heads stay zero).
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S_init = _f64(initial_state)
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    C = int(chunk_size)
    grp = Hv // Hq
    hv_list = list(range(Hv)) if heads is None else list(heads)
    seqs = sequences(B, T, cu_seqlens)
    out = {
        "o": np.zeros((B, T, Hv, V)),
        "final_state": np.zeros((len(seqs), Hv, K, V)),
        "Aqk": np.zeros((B, T, Hv, C)),
        "Akk": np.zeros((B, T, Hv, C)),
        "Akk_inv": np.zeros((B, T, Hv, C)),
        "W": np.zeros((B, T, Hv, K)),
        "U": np.zeros((B, T, Hv, V)),
        "G": np.zeros((B, T, Hv, K)),
        "QG": np.zeros((B, T, Hv, K)),
    }
    for n, (b, bos, eos) in enumerate(seqs):
        for hv in hv_list:
            hq = hv // grp
            S = np.zeros((K, V)) if S_init is None else S_init[n, hv].copy()
            for t0 in range(bos, eos, C):
                t1 = min(t0 + C, eos)
                L = t1 - t0
                q_c, k_c = q[b, t0:t1, hq], k[b, t0:t1, hq]
                v_c, g_c, b_c = v[b, t0:t1, hv], g[b, t0:t1, hv], beta[b, t0:t1, hv]
                G_c = chunk_local_cumsum(g_c)
                Aqk, Akk = intra_chunk_matrices(q_c, k_c, G_c, b_c, scale)
                Akk_inv = invert_unit_lower(Akk)
                W, U = recompute_w_u(Akk_inv, k_c, v_c, G_c, b_c)
                o_c, S = chunk_state_output(S, q_c, k_c, G_c, Aqk, W, U, scale)
                out["o"][b, t0:t1, hv] = o_c
                out["Aqk"][b, t0:t1, hv, :L] = Aqk
                out["Akk"][b, t0:t1, hv, :L] = Akk
                out["Akk_inv"][b, t0:t1, hv, :L] = Akk_inv
                out["W"][b, t0:t1, hv] = W
                out["U"][b, t0:t1, hv] = U
                out["G"][b, t0:t1, hv] = G_c
                out["QG"][b, t0:t1, hv] = gated_query(q_c, G_c)
            out["final_state"][n, hv] = S
    return out


# ---------------------------------------------------------------------------
# O3: varlen chunk metadata
# ---------------------------------------------------------------------------

def _check_chunk_size(chunk_size):
    # cuLA PR #135, review of tests/test_standalone_kernel_surface.py: a
    # chunk size of None, zero or below zero is rejected with ValueError.
    if chunk_size is None or isinstance(chunk_size, bool) or not isinstance(chunk_size, (int, np.integer)):
        raise ValueError("chunk_size must be a positive integer")
    if chunk_size <= 0:
        raise ValueError("chunk_size must be a positive integer")


def prepare_lens(cu_seqlens):
    """Sequence lengths cu[n+1] - cu[n] (cuLA PR #135, ``prepare_lens``)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    return cu[1:] - cu[:-1]


def prepare_chunk_indices(cu_seqlens, chunk_size):
    """(num_chunks, 2) pairs (sequence, chunk within sequence) and chunk offsets.

    cuLA PR #135 (cula/ops/kda/index.py review): the pairs have shape
    (num_chunks, 2) and the dtype of ``cu_seqlens``; empty input gives no
    chunks; an unsorted ``cu_seqlens`` is an error, not an empty result.
    ``offsets[n]`` is the number of chunks in sequences 0..n-1, so sequence n
    owns chunk ids offsets[n] .. offsets[n+1]-1.
    """
    _check_chunk_size(chunk_size)
    lens = prepare_lens(cu_seqlens)
    if np.any(lens < 0):
        raise ValueError("cu_seqlens must be non-decreasing")
    pairs = []
    offsets = [0]
    for n, ln in enumerate(lens.tolist()):
        nchunks = (ln + chunk_size - 1) // chunk_size
        for i in range(nchunks):
            pairs.append((n, i))
        offsets.append(offsets[-1] + nchunks)
    return (np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
            np.asarray(offsets, dtype=np.int32))


def num_chunks_bound(T, N, chunk_size):
    """Upper bound on the chunk count of N packed sequences of total length T."""
    return T // chunk_size + N if N > 0 else 0

