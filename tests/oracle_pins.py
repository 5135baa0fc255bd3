"""Checks that pin the fp64 oracle to facts the pages and the mathematics fix.

Each ``pin_*`` takes an oracle handle (``oracle.load(...)``) and raises
AssertionError when the oracle disagrees with the fact. They live in their own
module so that ``test_oracle_pins.py`` runs them on the oracle and
``test_oracle_mutants.py`` runs them on deliberately broken builds of it.

Page references (title, section):
  [KLA]  Gist.science, "Riepilogo Tecnico: Attenzione Lineare Kaczmarz (KLA)"
  [GN]   GeekNews, "Revisando las variantes de atencion lineal de la familia DeltaNet"
  [PB]   Paithon, "Scrivere meglio nella memoria: gate e delta rule"
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _one(x):
    """Add the B=1, H=1 axes: [T, ...] -> [1, T, 1, ...]."""
    x = np.asarray(x, dtype=np.float64)
    return x.reshape((1, x.shape[0], 1) + x.shape[1:])


def _run(orc, q, k, v, alpha, eta, eps, S0=None, **mode):
    """Single chain helper: q,k [T,dk], v [T,dv], alpha [T] or [T,dk], eta [T], S0 [dk,dv].
    ``mode``: beta_mode / q_scale of the oracle (KLA step and unscaled read by default)."""
    s0 = None if S0 is None else np.asarray(S0, dtype=np.float64)[None, None]
    o, ST = orc.recurrent(_one(q), _one(k), _one(v), _one(alpha), _one(eta), eps, s0, **mode)
    return o[0, :, 0], ST[0, 0]


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol:.1e} x {scale:.3g}"


# ----------------------------------------------------------------------------- pins
def pin_unrelaxed_constraint(orc):
    """[KLA] 'Derivazione Teorica' / 'Proprieta Chiave': with eta=1, eps=0 the write is the
    orthogonal projection onto {S : S^T k_t = v_t}, so re-reading with k_t returns v_t
    exactly, for any gate and any (unnormalised, nonzero) key."""
    rng = np.random.default_rng(11)
    T, dk, dv = 12, 8, 5
    for per_channel in (False, True):
        k = rng.normal(size=(T, dk)) * rng.uniform(0.2, 4.0, size=(T, 1))
        v = rng.normal(size=(T, dv))
        alpha = rng.uniform(0.3, 1.0, size=(T, dk) if per_channel else (T,))
        S0 = rng.normal(size=(dk, dv))
        o, _ = _run(orc, k, k, v, alpha, np.ones(T), 0.0, S0)
        _close(o, v, 1e-12, f"S_t^T k_t = v_t (per_channel={per_channel})")


def pin_deltanet_reread(orc):
    """[GN] 'DeltaNet': re-reading with the same unit key gives (1-beta) S~^T k + beta v;
    beta = 1 returns v exactly. With unit keys and eps=0 the KLA step is beta = eta."""
    rng = np.random.default_rng(12)
    dk, dv = 6, 4
    k = rng.normal(size=(1, dk))
    k /= np.linalg.norm(k)
    v = rng.normal(size=(1, dv))
    S0 = rng.normal(size=(dk, dv))
    o, _ = _run(orc, k, k, v, np.ones(1), np.ones(1), 0.0, S0)
    _close(o[0], v[0], 1e-12, "beta=1 re-read")
    o, _ = _run(orc, k, k, v, np.ones(1), np.full(1, 0.5), 0.0, S0)
    _close(o[0], 0.5 * (S0.T @ k[0]) + 0.5 * v[0], 1e-12, "beta=0.5 re-read")


def pin_pure_decay(orc):
    """[PB] 'Dimenticare: i gate' and [PB] 'Unire oblio e correzione': with the write
    switched off (eta = 0, so beta = 0) the memory only fades: S_t = alpha_t S_{t-1}.
    The printed example: factor 0.9 for ten steps leaves about 0.35."""
    g = _golden()["decay_ten_steps"]
    rng = np.random.default_rng(13)
    T, dk, dv = g["steps"], 5, 3
    S0 = rng.normal(size=(dk, dv))
    q = rng.normal(size=(T, dk))
    k = rng.normal(size=(T, dk))
    v = rng.normal(size=(T, dv))
    o, ST = _run(orc, q, k, v, np.full(T, g["alpha"]), np.zeros(T), 1e-6, S0)
    ratio = ST / S0
    _close(ratio, np.full_like(ratio, g["alpha"] ** T), 1e-13, "decay ratio")
    assert abs(float(ratio[0, 0]) - g["printed"]) <= g["printed_tolerance"], ratio[0, 0]
    for t in range(T):
        _close(o[t], g["alpha"] ** (t + 1) * (S0.T @ q[t]), 1e-12, f"decayed read t={t}")
    # per-key-channel gate: row i fades by prod_t alpha_t[i]
    a = rng.uniform(0.5, 1.0, size=(T, dk))
    _, ST = _run(orc, q, k, v, a, np.zeros(T), 1e-6, S0)
    _close(ST, np.prod(a, axis=0)[:, None] * S0, 1e-13, "per-channel decay")


def pin_orthogonal_locality(orc):
    """[GN] 'DeltaNet': the update is local in key space; reads along directions
    orthogonal to the current key are those of the decayed state."""
    rng = np.random.default_rng(14)
    dk, dv = 7, 5
    for per_channel in (False, True):
        k = rng.normal(size=(1, dk))
        u = rng.normal(size=dk)
        u -= (u @ k[0]) / (k[0] @ k[0]) * k[0]
        S0 = rng.normal(size=(dk, dv))
        alpha = rng.uniform(0.2, 1.0, size=(1, dk) if per_channel else (1,))
        eta = np.array([0.77])
        v = rng.normal(size=(1, dv))
        o, _ = _run(orc, u[None], k, v, alpha, eta, 1e-3, S0)
        D = alpha[0] if per_channel else np.full(dk, alpha[0])
        _close(o[0], (D[:, None] * S0).T @ u, 1e-12, f"orthogonal read (per_channel={per_channel})")


def pin_worked_scalar(orc):
    """[PB] 'Correggere: la delta rule': the phone-book numbers (7 -> 8.5 at half knob,
    -> 10 at full, stays 7 at zero, and the convex form 3.5 + 5 = 8.5)."""
    gd = _golden()
    for key in ("phone_book_half", "phone_book_full", "phone_book_zero"):
        g = gd[key]
        kk = np.array([[g["key"]]])
        o, ST = _run(orc, kk, kk, np.array([[g["value"]]]), np.ones(1), np.array([g["knob"]]), 0.0,
                     np.array([[g["state"]]]))
        assert abs(o[0, 0] - g["printed"]) <= 1e-12, (key, o[0, 0])
        assert abs(ST[0, 0] - g["printed"]) <= 1e-12, (key, ST[0, 0])
    c = gd["phone_book_convex"]
    half = gd["phone_book_half"]
    assert (1 - half["knob"]) * half["state"] == c["erase_part"]
    assert half["knob"] * half["value"] == c["write_part"]
    assert c["erase_part"] + c["write_part"] == c["printed"] == half["printed"]


def pin_marker_overshoot(orc):
    """[PB] 'Correggere: la delta rule' and 'Correggere' eigenvalue remark: a key of squared
    norm 2 at raw step 1 (KLA: eta = 2, eps = 0) has transition eigenvalue 1 - 2 = -1 along
    k, so the read oscillates 7 -> 13 -> 7 ...; the KLA step (eta = 1) lands on 10 at once."""
    g = _golden()["marker_overshoot"]
    n = len(g["printed_sequence"])
    kk = np.full((n, 1), np.sqrt(g["key_norm_sq"]))
    S0 = np.array([[g["state_read"] / np.sqrt(g["key_norm_sq"])]])
    v = np.full((n, 1), g["value"])
    eta = np.full(n, g["raw_beta"] * g["key_norm_sq"])
    o, _ = _run(orc, kk, kk, v, np.ones(n), eta, 0.0, S0)
    _close(o[:, 0], g["printed_sequence"], 1e-13, "overshoot sequence")
    o, _ = _run(orc, kk, kk, v, np.ones(n), np.ones(n), 0.0, S0)
    _close(o[:, 0], np.full(n, g["value"]), 1e-13, "KLA exact step")


def pin_transition_eigen(orc):
    """[PB] 'Correggere' and [GN] 'Transicion de estado estructurada': the transition
    I - beta k k^T has eigenvalue 1 - beta ||k||^2 along k and 1 on its orthogonal complement."""
    rng = np.random.default_rng(15)
    dk, dv = 6, 4
    k = rng.normal(size=dk) * 1.7
    u = rng.normal(size=dv)
    w = rng.normal(size=dk)
    w -= (w @ k) / (k @ k) * k
    eta = 1.7                           # beta ||k||^2 = 1.7 with eps = 0
    zero_v = np.zeros((1, dv))
    q = rng.normal(size=(1, dk))
    _, ST = _run(orc, q, k[None], zero_v, np.ones(1), np.array([eta]), 0.0, np.outer(k, u))
    _close(ST, (1 - eta) * np.outer(k, u), 1e-12, "eigenvalue along k")
    _, ST = _run(orc, q, k[None], zero_v, np.ones(1), np.array([eta]), 0.0, np.outer(w, u))
    _close(ST, np.outer(w, u), 1e-12, "eigenvalue 1 off k")


def pin_gradient_step(orc):
    """[PB] 'Tutto e regressione online', [GN] 'Derivacion desde la perdida de reconstruccion',
    [KLA] 'Proprieta Chiave': the write is one gradient step of L(S) = 1/2 ||S^T k - v||^2 taken
    from the decayed state with step beta = eta / (||k||^2 + eps). Gradient by central differences."""
    rng = np.random.default_rng(16)
    dk, dv = 4, 3
    k = rng.normal(size=dk)
    v = rng.normal(size=dv)
    S0 = rng.normal(size=(dk, dv))
    a, eta, eps = 0.8, 0.6, 0.25
    St = a * S0

    def L(S):
        r = S.T @ k - v
        return 0.5 * float(r @ r)

    grad = np.zeros_like(St)
    h = 1e-5
    for i in range(dk):
        for j in range(dv):
            Sp = St.copy()
            Sm = St.copy()
            Sp[i, j] += h
            Sm[i, j] -= h
            grad[i, j] = (L(Sp) - L(Sm)) / (2 * h)
    beta = eta / (k @ k + eps)
    _, ST = _run(orc, rng.normal(size=(1, dk)), k[None], v[None], np.array([a]), np.array([eta]), eps, S0)
    _close(ST, St - beta * grad, 1e-8, "gradient step")


def pin_linear_attention_split(orc):
    """[PB] 'Tutto e regressione online': with orthonormal keys the blind sum and the delta
    rule coincide only at full knob; at beta = 0.5 they differ by a factor two already after
    the first token. With orthonormal keys the prediction is always zero, so the delta-rule
    state is exactly half the accumulated sum of k v^T."""
    rng = np.random.default_rng(17)
    dk, dv, T = 5, 3, 5
    Q, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    K = Q.T[:T]                          # orthonormal rows
    V = rng.normal(size=(T, dv))
    _, S1 = _run(orc, K[:1], K[:1], V[:1], np.ones(1), np.full(1, 0.5), 0.0)
    _close(S1, 0.5 * np.outer(K[0], V[0]), 1e-13, "first token is half the blind write")
    _, ST = _run(orc, K, K, V, np.ones(T), np.full(T, 0.5), 0.0)
    _close(ST, 0.5 * K.T @ V, 1e-13, "half of the accumulated state")


def pin_dplr_transition(orc):
    """[GN] 'Transicion diagonal-bajo rango' and [PB] table row 'Gated DeltaNet': one step is
    S_t = A_t-form transition of the previous state plus beta k v^T, with A_t = D_t - b a^T,
    b = D_t k, a = beta k (page orientation). In the d_k x d_v orientation this reads
    S_t = (D_t - beta k (D_t k)^T) S_{t-1} + beta k v^T, and o_t = S_t^T q_t. Forgetting before
    predicting is what puts D_t on the right of the rank-one term."""
    rng = np.random.default_rng(18)
    T, dk, dv = 20, 6, 5
    for per_channel in (False, True):
        q = rng.normal(size=(T, dk))
        k = rng.normal(size=(T, dk)) * 1.3
        v = rng.normal(size=(T, dv))
        alpha = rng.uniform(0.4, 1.0, size=(T, dk) if per_channel else (T,))
        eta = rng.uniform(0.0, 1.5, size=T)
        eps = 0.3
        S = rng.normal(size=(dk, dv))
        o, ST = _run(orc, q, k, v, alpha, eta, eps, S)
        for t in range(T):
            D = np.diag(alpha[t] if per_channel else np.full(dk, alpha[t]))
            beta = eta[t] / (k[t] @ k[t] + eps)
            A_T = D - beta * np.outer(k[t], D @ k[t])
            S = A_T @ S + beta * np.outer(k[t], v[t])
            _close(o[t], S.T @ q[t], 1e-11, f"DPLR read t={t} per_channel={per_channel}")
        _close(ST, S, 1e-11, f"DPLR final state per_channel={per_channel}")


def pin_chunkwise_equals_recurrent(orc):
    """[GN] 'KDA por chunks': chunks of C tokens must give exactly the per-token state and
    outputs. The fp64 chunk algebra (oracle.chunkwise) must match the recurrence to rounding."""
    import oracle
    rng = np.random.default_rng(19)
    dk, dv = 6, 5
    for C in (1, 2, 4, 16):
        for T in (1, 15, 16, 17, 64):
            for per_channel in (False, True):
                q = rng.normal(size=(1, T, 2, dk))
                k = rng.normal(size=(1, T, 2, dk))
                v = rng.normal(size=(1, T, 2, dv))
                alpha = rng.uniform(0.5, 1.0, size=(1, T, 2, dk) if per_channel else (1, T, 2))
                eta = rng.uniform(0.0, 1.0, size=(1, T, 2))
                S0 = rng.normal(size=(1, 2, dk, dv))
                o_r, s_r = orc.recurrent(q, k, v, alpha, eta, 1e-6, S0)
                o_c, s_c = oracle.chunkwise(q, k, v, alpha, eta, 1e-6, S0, chunk=C)
                _close(o_c, o_r, 1e-12, f"chunkwise o C={C} T={T} pc={per_channel}")
                _close(s_c, s_r, 1e-12, f"chunkwise S C={C} T={T} pc={per_channel}")


def pin_continuation(orc):
    """The state is the whole carried context: running T1 tokens and then T2 tokens from the
    returned state equals one run of T1 + T2 tokens (same operations in the same order)."""
    rng = np.random.default_rng(20)
    T1, T2, dk, dv = 7, 9, 5, 4
    q = rng.normal(size=(1, T1 + T2, 3, dk))
    k = rng.normal(size=(1, T1 + T2, 3, dk))
    v = rng.normal(size=(1, T1 + T2, 3, dv))
    alpha = rng.uniform(0.5, 1.0, size=(1, T1 + T2, 3))
    eta = rng.uniform(0.0, 1.0, size=(1, T1 + T2, 3))
    S0 = rng.normal(size=(1, 3, dk, dv))
    o, S = orc.recurrent(q, k, v, alpha, eta, 1e-6, S0)
    o1, S1 = orc.recurrent(q[:, :T1], k[:, :T1], v[:, :T1], alpha[:, :T1], eta[:, :T1], 1e-6, S0)
    o2, S2 = orc.recurrent(q[:, T1:], k[:, T1:], v[:, T1:], alpha[:, T1:], eta[:, T1:], 1e-6, S1)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), o)
    assert np.array_equal(S2, S)


def pin_zero_key(orc):
    """Silent case, reading adopted: with k = 0 and eps = 0 the step beta := 0, so the token only
    applies the gate (no write)."""
    rng = np.random.default_rng(21)
    dk, dv = 4, 3
    S0 = rng.normal(size=(dk, dv))
    q = rng.normal(size=(1, dk))
    o, ST = _run(orc, q, np.zeros((1, dk)), rng.normal(size=(1, dv)), np.array([0.6]), np.array([0.9]), 0.0, S0)
    _close(ST, 0.6 * S0, 1e-15, "zero key state")
    _close(o[0], (0.6 * S0).T @ q[0], 1e-14, "zero key read")


def pin_raw_beta_worked(orc):
    """[PB] 'Correggere: la delta rule' read in the raw-beta mode (beta = eta, the write
    strength of DeltaNet and Gated DeltaNet): the phone-book numbers with a unit label
    (7 -> 8.5 at half knob, 10 at full, 7 at zero), and the marker label of squared norm 2
    at full knob overshooting 7 -> 13 -> 7 -> 13, where the KLA step lands on 10."""
    gd = _golden()
    for key in ("phone_book_half", "phone_book_full", "phone_book_zero"):
        g = gd[key]
        kk = np.array([[g["key"]]])
        o, ST = _run(orc, kk, kk, np.array([[g["value"]]]), np.ones(1), np.array([g["knob"]]), 0.3,
                     np.array([[g["state"]]]), beta_mode="raw")
        assert abs(o[0, 0] - g["printed"]) <= 1e-12, (key, o[0, 0])
        assert abs(ST[0, 0] - g["printed"]) <= 1e-12, (key, ST[0, 0])
    g = gd["marker_overshoot"]
    n = len(g["printed_sequence"])
    kk = np.full((n, 1), np.sqrt(g["key_norm_sq"]))
    S0 = np.array([[g["state_read"] / np.sqrt(g["key_norm_sq"])]])
    v = np.full((n, 1), g["value"])
    o, _ = _run(orc, kk, kk, v, np.ones(n), np.full(n, g["raw_beta"]), 0.0, S0, beta_mode="raw")
    _close(o[:, 0], g["printed_sequence"], 1e-13, "raw-beta overshoot sequence")
    o, _ = _run(orc, kk, kk, v, np.ones(n), np.full(n, g["raw_beta"]), 0.0, S0, beta_mode="kla")
    _close(o[:, 0], np.full(n, g["value"]), 1e-13, "KLA step on the same tokens")


def pin_raw_beta_first_write_and_limits(orc):
    """[PB] 'Tutto e regressione online': from an empty memory with the knob at half, the first
    write is half of what blind summing writes (S_1 = beta v k^T); [PB] 'Unire oblio e
    correzione': with beta -> 0 the write switches off with the correction and the memory only
    fades (S_t = alpha_t S_{t-1}), and with alpha = 1 the pure delta rule remains, whose
    re-read along a unit key is (1 - beta) S^T k + beta v."""
    rng = np.random.default_rng(31)
    dk, dv = 6, 4
    k = rng.normal(size=(1, dk))
    k /= np.linalg.norm(k)
    v = rng.normal(size=(1, dv))
    q = rng.normal(size=(1, dk))
    o, ST = _run(orc, q, k, v, np.ones(1), np.array([0.5]), 1e-3, None, beta_mode="raw")
    _close(ST, 0.5 * np.outer(k[0], v[0]), 1e-15, "first write at half knob")
    _close(o[0], 0.5 * (k[0] @ q[0]) * v[0], 1e-14, "first read at half knob")
    T = 5
    S0 = rng.normal(size=(dk, dv))
    a = rng.uniform(0.5, 1.0, size=T)
    qs = rng.normal(size=(T, dk))
    ks = rng.normal(size=(T, dk))
    o, ST = _run(orc, qs, ks, rng.normal(size=(T, dv)), a, np.zeros(T), 0.0, S0, beta_mode="raw")
    _close(ST, np.prod(a) * S0, 1e-13, "beta = 0 leaves only the fade")
    for t in range(T):
        _close(o[t], np.prod(a[: t + 1]) * (S0.T @ qs[t]), 1e-12, f"faded read t={t}")
    o, _ = _run(orc, k, k, v, np.ones(1), np.array([0.3]), 5.0, S0, beta_mode="raw")
    _close(o[0], 0.7 * (S0.T @ k[0]) + 0.3 * v[0], 1e-12, "pure delta rule re-read")


def pin_raw_beta_is_kla_with_rescaled_eta(orc):
    """Both step sizes write beta k e^T with the same residual, so the raw mode fed
    eta_t / (||k_t||^2 + eps) reproduces the KLA step fed eta_t, for any gate."""
    rng = np.random.default_rng(32)
    T, dk, dv = 9, 5, 4
    for per_channel in (False, True):
        q, k = rng.normal(size=(T, dk)), rng.normal(size=(T, dk)) * rng.uniform(0.3, 3.0, size=(T, 1))
        v = rng.normal(size=(T, dv))
        a = rng.uniform(0.4, 1.0, size=(T, dk) if per_channel else (T,))
        eta, eps = rng.uniform(0.1, 1.0, size=T), 0.25
        S0 = rng.normal(size=(dk, dv))
        o1, s1 = _run(orc, q, k, v, a, eta, eps, S0)
        o2, s2 = _run(orc, q, k, v, a, eta / (np.sum(k * k, axis=1) + eps), 123.0, S0, beta_mode="raw")
        _close(o2, o1, 1e-12, "raw vs KLA outputs")
        _close(s2, s1, 1e-12, "raw vs KLA states")


def pin_query_scale(orc):
    """[GN] 'Kimi Delta Attention': the read is o_t = S_t (d_k^{-1/2} q_t), and 'KDA por
    chunks' carries the same s in every read coefficient. From an empty state one token
    writes beta v k^T, so o_1 = s beta (k . q) v; the scale touches the read only."""
    rng = np.random.default_rng(33)
    dk, dv = 16, 3
    s = dk ** -0.5
    q, k, v = rng.normal(size=(1, dk)), rng.normal(size=(1, dk)), rng.normal(size=(1, dv))
    beta = 0.8 / (k[0] @ k[0] + 1e-2)
    o, ST = _run(orc, q, k, v, np.array([0.9]), np.array([0.8]), 1e-2, None, q_scale=s)
    _close(ST, beta * np.outer(k[0], v[0]), 1e-14, "one write from zero")
    _close(o[0], s * beta * (k[0] @ q[0]) * v[0], 1e-13, "scaled read of one write")
    T = 7
    q, k, v = rng.normal(size=(T, dk)), rng.normal(size=(T, dk)), rng.normal(size=(T, dv))
    a, eta = rng.uniform(0.5, 1.0, size=(T, dk)), rng.uniform(0.1, 1.0, size=T)
    S0 = rng.normal(size=(dk, dv))
    o1, s1 = _run(orc, q, k, v, a, eta, 1e-3, S0)
    o2, s2 = _run(orc, q, k, v, a, eta, 1e-3, S0, q_scale=s)
    _close(o2, s * o1, 1e-13, "outputs scale with s")
    _close(s2, s1, 0.0, "state does not see s")


def pin_backward_finite_differences(orc):
    """The backward pass is the derivative of the forward: for L = sum(W_o * o) + sum(W_s * S_T)
    with random weights, every gradient the backward returns (q, k, v, alpha, eta, S0) matches
    central differences of the forward oracle, for both gates, both step sizes, a query scale,
    with and without a final-state gradient."""
    rng = np.random.default_rng(41)
    B, T, H, dk, dv = 1, 6, 1, 3, 2
    names = {"q": "dq", "k": "dk", "v": "dv", "alpha": "dalpha", "eta": "deta", "S0": "dS0"}
    for per_channel, mode, with_ds in ((False, "kla", True), (True, "kla", False), (False, "raw", False),
                                       (True, "raw", True)):
        x = {"q": rng.normal(size=(B, T, H, dk)), "k": rng.normal(size=(B, T, H, dk)) * 0.7,
             "v": rng.normal(size=(B, T, H, dv)),
             "alpha": rng.uniform(0.5, 1.0, size=(B, T, H, dk) if per_channel else (B, T, H)),
             "eta": rng.uniform(0.1, 0.9, size=(B, T, H)), "S0": rng.normal(size=(B, H, dk, dv))}
        Wo, Ws = rng.normal(size=(B, T, H, dv)), (rng.normal(size=(B, H, dk, dv)) if with_ds else None)
        eps, s = 0.3, 0.7

        def loss(a):
            o, ST = orc.recurrent(a["q"], a["k"], a["v"], a["alpha"], a["eta"], eps, a["S0"], beta_mode=mode,
                                  q_scale=s)
            return float(np.sum(o * Wo) + (np.sum(ST * Ws) if Ws is not None else 0.0))
        g = orc.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], eps, x["S0"], Wo, Ws, beta_mode=mode,
                         q_scale=s)
        for n, arr in x.items():
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                xp, xm = dict(x), dict(x)
                xp[n] = arr.copy()
                xm[n] = arr.copy()
                xp[n][idx] += 1e-6
                xm[n][idx] -= 1e-6
                fd[idx] = (loss(xp) - loss(xm)) / 2e-6
            _close(g[names[n]], fd, 1e-7, f"d{n} ({mode}, per_channel={per_channel})")


PINS = [
    pin_unrelaxed_constraint, pin_deltanet_reread, pin_pure_decay, pin_orthogonal_locality,
    pin_worked_scalar, pin_marker_overshoot, pin_transition_eigen, pin_gradient_step,
    pin_linear_attention_split, pin_dplr_transition, pin_chunkwise_equals_recurrent,
    pin_continuation, pin_zero_key, pin_raw_beta_worked, pin_raw_beta_first_write_and_limits,
    pin_raw_beta_is_kla_with_rescaled_eta, pin_query_scale, pin_backward_finite_differences,
]
