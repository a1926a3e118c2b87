"""Plant plausible mistakes in the oracle and check that its pins catch each one.

Every mutation below is applied to the oracle module on the CPU (monkeypatch)
and must make at least one pin of ``test_oracle.py`` fail.  This is the
evidence that the pins constrain the oracle, not just agree with it.
"""

import numpy as np
import pytest

import tests.test_oracle as pins
from oracle import kda_ref as ref

PIN_CALLS = [
    pins.test_scalar_recurrence_hand_worked,
    pins.test_vector_recurrence_hand_worked,
    lambda: pins.test_chunked_equals_recurrent(16, 37),
    lambda: pins.test_chunked_equals_recurrent(64, 130),
    pins.test_chunked_equals_recurrent_varlen_gva,
    pins.test_inverse_is_inverse,
    pins.test_intra_matrices_brute_force_products_of_gates,
    pins.test_w_u_solve_the_triangular_systems,
    pins.test_beta_zero_is_pure_gated_decay,
    pins.test_orthonormal_keys_store_and_retrieve,
    pins.test_rewrite_same_key_overwrites_value,
    pins.test_gva_equals_mha_with_repeated_qk,
    pins.test_continuation_across_calls,
    lambda: pins.test_chunk_indices_brute_force([1, 63, 64, 65, 0, 129, 3], 64),
    pins.test_gated_query_closed_form_constant_gates,
    pins.test_gated_query_brute_force_products,
]


def _failing_pins():
    failed = 0
    for call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            failed += 1
    return failed


_orig = {name: getattr(ref, name) for name in (
    "chunk_local_cumsum", "intra_chunk_matrices", "invert_unit_lower",
    "recompute_w_u", "chunk_state_output", "kda_recurrent", "prepare_chunk_indices", "gated_query")}


def _exclusive_cumsum(g):
    return np.cumsum(g, axis=0) - g


def _aqk_no_diagonal(q, k, G, beta, scale):
    Aqk, Akk = _orig["intra_chunk_matrices"](q, k, G, beta, scale)
    return np.tril(Aqk, -1), Akk


def _akk_no_beta(q, k, G, beta, scale):
    Aqk, Akk = _orig["intra_chunk_matrices"](q, k, G, beta, scale)
    return Aqk, Akk / np.where(beta[:, None] == 0, 1, beta[:, None])


def _akk_beta_on_columns(q, k, G, beta, scale):
    Aqk, Akk = _orig["intra_chunk_matrices"](q, k, G, beta, scale)
    raw = Akk / np.where(beta[:, None] == 0, 1, beta[:, None])
    return Aqk, raw * beta[None, :]


def _akk_sign_flipped(q, k, G, beta, scale):
    Aqk, Akk = _orig["intra_chunk_matrices"](q, k, G, beta, scale)
    return Aqk, -Akk


def _inverse_first_order(A):
    return np.eye(A.shape[-1]) - A


def _inverse_transposed(A):
    return np.swapaxes(_orig["invert_unit_lower"](A), -1, -2)


def _w_without_gate(X, k, v, G, beta):
    return X @ (beta[:, None] * k), X @ (beta[:, None] * v)


def _u_without_beta(X, k, v, G, beta):
    W, _ = _orig["recompute_w_u"](X, k, v, G, beta)
    return W, X @ v


def _delta_sign(S0, q, k, G, Aqk, W, U, scale):
    return _orig["chunk_state_output"](S0, q, k, G, Aqk, -W, U, scale)


def _decay_with_first_row(S0, q, k, G, Aqk, W, U, scale):
    G2 = G.copy()
    G2[-1] = G[0]
    o, _ = _orig["chunk_state_output"](S0, q, k, G, Aqk, W, U, scale)
    _, S1 = _orig["chunk_state_output"](S0, q, k, G2, Aqk, W, U, scale)
    return o, S1


def _aqk_transposed(S0, q, k, G, Aqk, W, U, scale):
    return _orig["chunk_state_output"](S0, q, k, G, Aqk.T, W, U, scale)


def _recurrent_decay_after_update(q, k, v, g, beta, scale, initial_state=None,
                                  cu_seqlens=None, heads=None):
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    grp = Hv // Hq
    seqs = ref.sequences(B, T, cu_seqlens)
    o = np.zeros((B, T, Hv, V))
    fin = np.zeros((len(seqs), Hv, K, V))
    for n, (b, s, e) in enumerate(seqs):
        for hv in range(Hv):
            S = np.zeros((K, V)) if initial_state is None else np.array(initial_state[n, hv], float)
            for t in range(s, e):
                kt, qt = k[b, t, hv // grp], q[b, t, hv // grp]
                S = S + beta[b, t, hv] * np.outer(kt, v[b, t, hv] - kt @ S)
                S = np.exp(g[b, t, hv])[:, None] * S
                o[b, t, hv] = scale * S.T @ qt
            fin[n, hv] = S
    return o, fin


def _qg_negated_gate(q_c, G_c):
    return q_c * np.exp(-G_c)


def _qg_previous_row(q_c, G_c):
    return _orig["gated_query"](q_c, _exclusive_cumsum(np.diff(G_c, axis=0, prepend=0.0)))


def _qg_scaled(q_c, G_c):
    return _orig["gated_query"](q_c, G_c) * q_c.shape[-1] ** -0.5


def _indices_floor(cu, C):
    lens = ref.prepare_lens(cu)
    pairs, off = [], [0]
    for n, ln in enumerate(lens.tolist()):
        for i in range(ln // C):
            pairs.append((n, i))
        off.append(off[-1] + ln // C)
    return np.asarray(pairs, np.int32).reshape(-1, 2), np.asarray(off, np.int32)


MUTATIONS = {
    "exclusive cumsum": ("chunk_local_cumsum", _exclusive_cumsum),
    "Aqk without its diagonal": ("intra_chunk_matrices", _aqk_no_diagonal),
    "Akk without beta": ("intra_chunk_matrices", _akk_no_beta),
    "beta on Akk columns": ("intra_chunk_matrices", _akk_beta_on_columns),
    "Akk sign flipped": ("intra_chunk_matrices", _akk_sign_flipped),
    "first-order inverse": ("invert_unit_lower", _inverse_first_order),
    "transposed inverse": ("invert_unit_lower", _inverse_transposed),
    "W without the gate": ("recompute_w_u", _w_without_gate),
    "U without beta": ("recompute_w_u", _u_without_beta),
    "Delta = U + W S": ("chunk_state_output", _delta_sign),
    "state decays with the first row": ("chunk_state_output", _decay_with_first_row),
    "Aqk transposed": ("chunk_state_output", _aqk_transposed),
    "recurrence decays after the update": ("kda_recurrent", _recurrent_decay_after_update),
    "chunk count rounds down": ("prepare_chunk_indices", _indices_floor),
    "QG with the gate negated": ("gated_query", _qg_negated_gate),
    "QG with the previous row's cumsum": ("gated_query", _qg_previous_row),
    "QG carrying scale": ("gated_query", _qg_scaled),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(ref, attr, fn)
    assert _failing_pins() >= 1, f"no pin caught the planted mistake: {name}"


def test_pins_pass_unmutated():
    assert _failing_pins() == 0
