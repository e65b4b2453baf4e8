"""Pins for the FP64 oracle: checks against what the source pages and the
mathematics fix, independent of the oracle's own code.

Each pin is a plain function ``pin_*(fwd)`` that raises AssertionError on a
mismatch; ``fwd`` is an oracle entry point, so the same pins also run against
deliberately broken copies of the oracle (test_pins_catch_planted_mistakes)
to show that a plausible mistake anywhere in it fails at least one pin.

Sources:
* FlashInfer docs, "flashinfer.gdn2_prefill.chunk_gated_delta_rule2": the
  recurrence (op description), the reduction to scalar GDN with channel-
  constant g and w == beta, gate defaults and the scale default (parameters).
* burn-gdn2 README, "Per-token recurrence": the product form
  S_t = (I - k_t (b_t * k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t * v_t)^T.
* FlashGDN-2 README, "Quick start": prefill then decode from the carried state.
"""
import os
import shutil

import numpy as np
import pytest

import oracle

RTOL = 1e-12  # fp64 against fp64 arithmetic of a different form


def rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def close(a, b, tol=RTOL, what=""):
    e = rel_err(a, b)
    assert e <= tol, "%s: relative error %.3e > %.1e" % (what, e, tol)


def rand_case(rng, T, H=1, HV=1, K=5, V=4, g_max=0.5, beta_max=1.0, h0=True, unit_k=False):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, HV, V))
    g = -g_max * rng.random((T, HV, K))
    beta = beta_max * rng.random((T, HV, K))
    w = rng.random((T, HV, V))
    S0 = 0.3 * rng.standard_normal((1, HV, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, w=w, initial_state=S0)


# --------------------------------------------------------------------------
# P1: brute force of the burn-gdn2 product form, T <= 8.  The final state is
# expanded explicitly as  S_T = M_T ... M_1 S_0 + sum_s M_T ... M_{s+1} k_s (w_s v_s)^T
# with M_t = (I - k_t (b_t k_t)^T) diag(exp g_t); outputs use the same
# expansion up to each t.  Pins decay order, erase (incl. beta placement),
# write gate, scale and the read-after-write output.
# --------------------------------------------------------------------------
def _product_form(c, scale):
    q, k, v, g, b, w = (c[x][:, 0] for x in ("q", "k", "v", "g", "beta", "w"))
    S0 = c["initial_state"][0, 0] if c["initial_state"] is not None else np.zeros((k.shape[1], v.shape[1]))
    T, K = k.shape
    Ms = [(np.eye(K) - np.outer(k[t], b[t] * k[t])) @ np.diag(np.exp(g[t])) for t in range(T)]
    outs, states = [], []
    for t in range(T):
        P = np.eye(K)
        for r in range(t, -1, -1):
            P = P @ Ms[r]
        S = P @ S0
        for s in range(t + 1):
            Pr = np.eye(K)
            for r in range(t, s, -1):
                Pr = Pr @ Ms[r]
            S = S + Pr @ np.outer(k[s], w[s] * v[s])
        states.append(S)
        outs.append(scale * q[t] @ S)
    return np.array(outs), states[-1]


def pin_brute_force(fwd):
    rng = np.random.default_rng(11)
    for T in (1, 2, 5, 8):
        for K, V in ((4, 3), (3, 5)):
            c = rand_case(rng, T, K=K, V=V, beta_max=2.0)
            o, hT = fwd(**c, scale=0.7)
            o_ref, S_ref = _product_form(c, 0.7)
            close(o[:, 0], o_ref, what="brute-force o T=%d" % T)
            close(hT[0, 0], S_ref, what="brute-force state T=%d" % T)


# --------------------------------------------------------------------------
# P2: reduction to the scalar gated delta rule (FlashInfer docs): channel-
# constant g = log(alpha_t), beta = w = b_t give the textbook update
# S_t = alpha_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T.
# --------------------------------------------------------------------------
def pin_scalar_gdn(fwd):
    rng = np.random.default_rng(12)
    T, K, V = 40, 6, 5
    q = rng.standard_normal((T, 1, K)); k = rng.standard_normal((T, 1, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, V))
    alpha = rng.uniform(0.5, 1.0, T); b = rng.uniform(0.0, 1.0, T)
    S0 = rng.standard_normal((1, 1, K, V))
    g = np.log(alpha)[:, None, None] * np.ones((T, 1, K))
    beta = b[:, None, None] * np.ones((T, 1, K))
    w = b[:, None, None] * np.ones((T, 1, V))
    o, hT = fwd(q, k, v, g, beta, w, scale=0.5, initial_state=S0)
    S = S0[0, 0].copy()
    for t in range(T):
        kt = k[t, 0]
        S = alpha[t] * (np.eye(K) - b[t] * np.outer(kt, kt)) @ S + b[t] * np.outer(kt, v[t, 0])
        close(o[t, 0], 0.5 * q[t, 0] @ S, what="scalar GDN o")
    close(hT[0, 0], S, what="scalar GDN state")


# --------------------------------------------------------------------------
# P3: g = 0, beta = 0, w = 1 is causal linear attention:
# O = scale (tril(Q K^T) V + Q S_0),  S_T = S_0 + K^T V  (one matmul each).
# --------------------------------------------------------------------------
def pin_linear_attention(fwd):
    rng = np.random.default_rng(13)
    T, K, V = 70, 8, 6
    c = rand_case(rng, T, K=K, V=V)
    o, hT = fwd(c["q"], c["k"], c["v"], np.zeros((T, 1, K)), np.zeros((T, 1, K)),
                np.ones((T, 1, V)), scale=0.25, initial_state=c["initial_state"])
    Q, Kk, Vv, S0 = c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], c["initial_state"][0, 0]
    close(o[:, 0], 0.25 * (np.tril(Q @ Kk.T) @ Vv + Q @ S0), what="linear attention o")
    close(hT[0, 0], S0 + Kk.T @ Vv, what="linear attention state")


# --------------------------------------------------------------------------
# P4: one token, closed form.  D = diag(exp g); u = w v - S_0^T D (beta k);
# S_1 = D S_0 + k u^T;  o = scale (q^T D S_0 + (q . k) u).  With S_0 = 0:
# o = scale (q . k) (w v).
# --------------------------------------------------------------------------
def pin_single_token(fwd):
    rng = np.random.default_rng(14)
    for h0 in (True, False):
        c = rand_case(rng, 1, K=7, V=5, beta_max=2.0, h0=h0)
        o, hT = fwd(**c, scale=0.9)
        q, k, v, g, b, w = (c[x][0, 0] for x in ("q", "k", "v", "g", "beta", "w"))
        D = np.diag(np.exp(g))
        if h0:
            S0 = c["initial_state"][0, 0]
            u = w * v - S0.T @ D @ (b * k)
            close(hT[0, 0], D @ S0 + np.outer(k, u), what="single-token state")
            close(o[0, 0], 0.9 * (q @ D @ S0 + (q @ k) * u), what="single-token o")
        else:
            close(o[0, 0], 0.9 * (q @ k) * (w * v), what="single-token o (zero state)")
            close(hT[0, 0], np.outer(k, w * v), what="single-token state (zero state)")


# --------------------------------------------------------------------------
# P5: split sequence with carried state equals one pass (FlashGDN-2 quick
# start: prefill, then continue from the returned state).
# --------------------------------------------------------------------------
def pin_split_sequence(fwd):
    rng = np.random.default_rng(15)
    T = 130
    c = rand_case(rng, T, H=1, HV=2, K=6, V=5, beta_max=2.0)
    c["initial_state"] = 0.3 * rng.standard_normal((1, 2, 6, 5))
    o, hT = fwd(**c, scale=0.6)
    for t in (1, 63, 64, 65, T - 1):
        a = {x: (None if c[x] is None else c[x][:t]) for x in ("q", "k", "v", "g", "beta", "w")}
        b = {x: (None if c[x] is None else c[x][t:]) for x in ("q", "k", "v", "g", "beta", "w")}
        o1, h1 = fwd(**a, initial_state=c["initial_state"], scale=0.6)
        o2, h2 = fwd(**b, initial_state=h1, scale=0.6)
        close(np.concatenate([o1, o2]), o, what="split at %d: o" % t)
        close(h2, hT, what="split at %d: state" % t)


# --------------------------------------------------------------------------
# P6: delta-write invariant.  With beta = 1 and ||k_t|| = 1 the recurrence
# gives k_t^T S_t = w_t * v_t exactly (the new state stores the gated value
# under key k_t).
# --------------------------------------------------------------------------
def pin_delta_write(fwd):
    rng = np.random.default_rng(16)
    T, K, V = 9, 6, 4
    c = rand_case(rng, T, K=K, V=V, unit_k=True)
    c["beta"] = np.ones((T, 1, K))
    for t in range(1, T + 1):
        sub = {x: c[x][:t] for x in ("q", "k", "v", "g", "beta", "w")}
        _, h = fwd(**sub, initial_state=c["initial_state"])
        close(c["k"][t - 1, 0] @ h[0, 0], c["w"][t - 1, 0] * c["v"][t - 1, 0], tol=1e-11,
              what="delta write t=%d" % t)


# --------------------------------------------------------------------------
# P7: beta = 0 (decay only, GLA-like): with the global inclusive cumsum G,
# o_t = scale [ (q_t e^{G_t})^T S_0 + sum_{s<=t} ((q_t e^{G_t - G_s}) . k_s) (w_s v_s) ]
# and S_T = e^{G_T} S_0 + sum_s (k_s e^{G_T - G_s}) (w_s v_s)^T.
# --------------------------------------------------------------------------
def pin_decay_only(fwd):
    rng = np.random.default_rng(17)
    T, K, V = 30, 5, 4
    c = rand_case(rng, T, K=K, V=V, g_max=0.4)
    c["beta"] = np.zeros((T, 1, K))
    o, hT = fwd(**c, scale=0.8)
    q, k, v, g, w = (c[x][:, 0] for x in ("q", "k", "v", "g", "w"))
    S0 = c["initial_state"][0, 0]
    G = np.cumsum(g, axis=0)
    for t in range(T):
        ref = (q[t] * np.exp(G[t])) @ S0
        for s in range(t + 1):
            ref = ref + np.dot(q[t] * np.exp(G[t] - G[s]), k[s]) * (w[s] * v[s])
        close(o[t, 0], 0.8 * ref, what="decay-only o t=%d" % t)
    S = np.exp(G[-1])[:, None] * S0
    for s in range(T):
        S = S + np.outer(k[s] * np.exp(G[-1] - G[s]), w[s] * v[s])
    close(hT[0, 0], S, what="decay-only state")


# --------------------------------------------------------------------------
# P8: structure.
# --------------------------------------------------------------------------
def pin_packing(fwd):
    """Packed varlen input equals separate calls per sequence; an empty
    sequence returns its initial state."""
    rng = np.random.default_rng(18)
    lens = [5, 0, 17, 1, 9]
    T = sum(lens)
    c = rand_case(rng, T, H=1, HV=2, K=4, V=3, beta_max=2.0)
    S0 = rng.standard_normal((len(lens), 2, 4, 3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, hT = fwd(**{**c, "initial_state": S0}, cu_seqlens=cu, scale=0.5)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        sub = {x: c[x][sl] for x in ("q", "k", "v", "g", "beta", "w")}
        o_n, h_n = fwd(**sub, initial_state=S0[n:n + 1], scale=0.5)
        if lens[n]:
            close(o[sl], o_n, what="packing o seq %d" % n)
        close(hT[n], h_n[0], what="packing state seq %d" % n)
    close(hT[1], S0[1], tol=0.0, what="empty sequence keeps its state")


def pin_grouped_heads(fwd):
    """HV = 4 value heads on H = 2 key heads equals H = HV with q/k expanded
    so that value head hv reads key head hv // (HV / H)."""
    rng = np.random.default_rng(19)
    T, H, HV, K, V = 12, 2, 4, 4, 3
    c = rand_case(rng, T, H=H, HV=HV, K=K, V=V)
    S0 = rng.standard_normal((1, HV, K, V))
    o, hT = fwd(**{**c, "initial_state": S0}, scale=0.5)
    idx = np.arange(HV) // (HV // H)
    o2, h2 = fwd(**{**c, "q": c["q"][:, idx], "k": c["k"][:, idx], "initial_state": S0}, scale=0.5)
    close(o, o2, what="GVA o")
    close(hT, h2, what="GVA state")
    # and it really is head hv // 2, not hv % 2
    o3, _ = fwd(**{**c, "q": c["q"][:, np.arange(HV) % H], "k": c["k"][:, np.arange(HV) % H],
                   "initial_state": S0}, scale=0.5)
    assert rel_err(o, o3) > 1e-3, "GVA head map is not distinguishable"


def pin_head_counts(fwd):
    """The FlashInfer docs' head counts: HK equals H or HV, and H, HV are
    equal or one a multiple of the other; one state per state head hs < HS =
    max(H, HV), which reads q head hs // (HS / H), k head hs // (HS / HK) and
    v head hs // (HS / HV).  Each case equals H = HK = HV = HS with q, k, v
    expanded by those maps; a map taken modulo the head count is
    distinguishable."""
    rng = np.random.default_rng(25)
    T, K, V = 13, 4, 3
    for H, HK, HV in ((4, 2, 2), (4, 4, 2), (2, 4, 4), (2, 2, 4), (3, 3, 6), (6, 2, 2)):
        HS = max(H, HV)
        q = rng.standard_normal((T, H, K))
        k = rng.standard_normal((T, HK, K))
        v = rng.standard_normal((T, HV, V))
        g = -0.5 * rng.random((T, HS, K))
        beta = rng.random((T, HS, K))
        w = rng.random((T, HS, V))
        S0 = rng.standard_normal((1, HS, K, V))
        o, hT = fwd(q, k, v, g, beta, w, initial_state=S0, scale=0.5)
        assert o.shape == (T, HS, V) and hT.shape == (1, HS, K, V)
        iq, ik, iv = (np.arange(HS) // (HS // n) for n in (H, HK, HV))
        o2, h2 = fwd(q[:, iq], k[:, ik], v[:, iv], g, beta, w, initial_state=S0, scale=0.5)
        close(o, o2, what="heads %s o" % ((H, HK, HV),))
        close(hT, h2, what="heads %s state" % ((H, HK, HV),))
        for n, arr, pos in ((H, q, 0), (HK, k, 1), (HV, v, 2)):
            if n == HS:
                continue
            mod = [q[:, iq], k[:, ik], v[:, iv]]
            mod[pos] = arr[:, np.arange(HS) % n]
            o3, _ = fwd(*mod, g, beta, w, initial_state=S0, scale=0.5)
            assert rel_err(o, o3) > 1e-3, "head map of tensor %d not distinguishable at %s" % (pos, (H, HK, HV))


def pin_l2norm(fwd):
    """The fused q/k L2 norm equals pre-normalised input; it is a no-op on
    unit rows."""
    rng = np.random.default_rng(20)
    c = rand_case(rng, 10, K=6, V=4)
    c["q"] *= 3.0; c["k"] *= 0.2
    o1, h1 = fwd(**c, use_qk_l2norm=True, scale=0.5)
    qn = c["q"] / np.linalg.norm(c["q"], axis=-1, keepdims=True)
    kn = c["k"] / np.linalg.norm(c["k"], axis=-1, keepdims=True)
    o2, h2 = fwd(**{**c, "q": qn, "k": kn}, scale=0.5)
    close(o1, o2, what="l2norm o"); close(h1, h2, what="l2norm state")


def pin_channel_permutations(fwd):
    """Value channels evolve independently: permuting V columns of v, w, S_0
    permutes o and S columns.  Permuting key channels of q, k, g, beta and
    S_0 rows leaves o unchanged and permutes S rows."""
    rng = np.random.default_rng(21)
    c = rand_case(rng, 20, K=5, V=6, beta_max=2.0)
    o, hT = fwd(**c, scale=0.5)
    pv = rng.permutation(6)
    o2, h2 = fwd(**{**c, "v": c["v"][..., pv], "w": c["w"][..., pv],
                    "initial_state": c["initial_state"][..., pv]}, scale=0.5)
    close(o2, o[..., pv], what="V permutation o"); close(h2, hT[..., pv], what="V permutation S")
    pk = rng.permutation(5)
    o3, h3 = fwd(**{**c, "q": c["q"][..., pk], "k": c["k"][..., pk], "g": c["g"][..., pk],
                    "beta": c["beta"][..., pk], "initial_state": c["initial_state"][:, :, pk]},
                 scale=0.5)
    close(o3, o, what="K permutation o"); close(h3, hT[:, :, pk], what="K permutation S")


def pin_defaults(fwd):
    """Missing gates mean g = 0, beta = 1, w = 1; scale <= 0 or None means
    1/sqrt(K) (FlashInfer docs, parameters)."""
    rng = np.random.default_rng(22)
    c = rand_case(rng, 11, K=9, V=4)
    T = 11
    o1, h1 = fwd(c["q"], c["k"], c["v"], initial_state=c["initial_state"])
    o2, h2 = fwd(c["q"], c["k"], c["v"], np.zeros((T, 1, 9)), np.ones((T, 1, 9)),
                 np.ones((T, 1, 4)), scale=1.0 / 3.0, initial_state=c["initial_state"])
    close(o1, o2, what="defaults o"); close(h1, h2, what="defaults S")
    o3, _ = fwd(c["q"], c["k"], c["v"], scale=0.0, initial_state=c["initial_state"])
    close(o3, o2, what="scale 0 -> 1/sqrt(K)")


PINS = [pin_brute_force, pin_scalar_gdn, pin_linear_attention, pin_single_token,
        pin_split_sequence, pin_delta_write, pin_decay_only, pin_packing,
        pin_grouped_heads, pin_head_counts, pin_l2norm, pin_channel_permutations, pin_defaults]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.gdn2_forward)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(23)
    c = rand_case(rng, 50, H=2, HV=4, K=6, V=5)
    c["initial_state"] = rng.standard_normal((1, 4, 6, 5))
    o1, h1 = oracle.gdn2_forward(**c, threads=1)
    o4, h4 = oracle.gdn2_forward(**c, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(h1, h4)


def test_units_subset():
    """Computing a subset of (n, hv) units gives the same rows as the full run."""
    rng = np.random.default_rng(24)
    lens = [7, 12]
    c = rand_case(rng, 19, H=1, HV=3, K=4, V=4)
    S0 = rng.standard_normal((2, 3, 4, 4))
    cu = [0, 7, 19]
    o, hT = oracle.gdn2_forward(**{**c, "initial_state": S0}, cu_seqlens=cu)
    o_s, h_s = oracle.gdn2_forward(**{**c, "initial_state": S0}, cu_seqlens=cu, units=[(1, 2)])
    assert np.array_equal(o_s[7:19, 2], o[7:19, 2])
    assert np.array_equal(h_s[1, 2], hT[1, 2])
    assert np.isnan(o_s[:7]).all() and np.isnan(h_s[0]).all()


# --------------------------------------------------------------------------
# Planted mistakes: each mutant is a copy of the oracle's C source with one
# plausible error; the pins above must reject every one of them.
# --------------------------------------------------------------------------
MUTANTS = {
    "erase_sign": ("u[j] = (w ? w[j] : 1.0) * vv[j] - u[j];", "u[j] = (w ? w[j] : 1.0) * vv[j] + u[j];"),
    "erase_without_beta": ("const double bk = (b ? b[c] : 1.0) * kt[c];", "const double bk = kt[c];"),
    "write_gate_dropped": ("u[j] = (w ? w[j] : 1.0) * vv[j] - u[j];", "u[j] = vv[j] - u[j];"),
    "decay_sign": ("const double a = exp(g[c]);", "const double a = exp(-g[c]);"),
    "head_map_modulo": ("const int hq = hs / (HS / H);", "const int hq = hs % H;"),
    "k_head_map_modulo": ("const int hk = hs / (HS / HK);", "const int hk = hs % HK;"),
    "v_head_map_modulo": ("const int hvv = hs / (HS / HV);", "const int hvv = hs % HV;"),
    "write_with_q": ("row[j] += kt[c] * u[j];", "row[j] += qt[c] * u[j];"),
    "scale_dropped": ("for (j = 0; j < V; j++) o[j] *= J->scale;", ""),
    "l2_dropped": ("for (i = 0; i < n; i++) y[i] = x[i] / d;", "for (i = 0; i < n; i++) y[i] = x[i];"),
    "initial_state_ignored": ("if (J->h0) memcpy(", "if (0) memcpy("),
    "beta_default_zero": ("(b ? b[c] : 1.0)", "(b ? b[c] : 0.0)"),
    "output_before_write": None,   # block move, built below
    "decay_after_erase": None,     # block move, built below
}


def _block(src, start_marker, end_marker):
    i = src.index(start_marker)
    j = src.index(end_marker, i)
    return i, j


def _mutant_source(name, src):
    rep = MUTANTS[name]
    if rep is not None:
        assert rep[0] in src, name
        return src.replace(rep[0], rep[1], 1)
    if name == "output_before_write":
        i, j = _block(src, "/* write: S <- S + k_t u^T */", "/* output after the write")
        k2 = src.index("    }\n    memcpy(J->hT", j)
        write_blk, out_blk = src[i:j], src[j:k2]
        return src[:i] + out_blk + "        " + write_blk.strip() + "\n" + src[k2:]
    if name == "decay_after_erase":
        i, j = _block(src, "/* decay: S <- diag(exp(g_t)) S */", "/* erase read on the decayed state")
        k2 = src.index("/* write: S <- S + k_t u^T */", j)
        decay_blk, erase_blk = src[i:j], src[j:k2]
        return src[:i] + erase_blk + decay_blk + "        " + src[k2:]
    raise KeyError(name)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn2_oracle.c")).read()
    msrc = _mutant_source(name, src)
    assert msrc != src
    p = tmp_path / ("m_%s.c" % name)
    p.write_text(msrc)
    lib = oracle.load_library(oracle.compile_c(str(p), str(tmp_path / ("m_%s.so" % name))))

    def fwd(*a, **kw):
        return oracle.gdn2_forward(*a, lib=lib, **kw)

    failed = []
    for pin in PINS:
        try:
            pin(fwd)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
