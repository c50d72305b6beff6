"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

None of these tests re-types the oracle's token loop.  Each checks the
oracle against something else: an explicit product of per-token transition
matrices (brute-force unrolling), closed forms for special inputs, literal
constants, and invariants (chaining, packing, normalisation).  A plausible
mistake in the oracle -- a dropped term, a flipped sign, read-before-write,
a transposed state, a wrong gate -- fails at least one of them.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

BIG = 1.0e4          # logit with sigmoid exactly 1.0 (or 0.0 for -BIG) in fp64


def rand_problem(rng, T, H, D, N=None, lengths=None, lb=-5.0, zero_state=False):
    if lengths is None:
        lengths = [T]
    N = len(lengths)
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    p = dict(
        q=rng.standard_normal((T, H, D)), k=rng.standard_normal((T, H, D)),
        v=rng.standard_normal((T, H, D)), g=rng.standard_normal((T, H, D)),
        beta=rng.standard_normal((T, H)),
        A_log=np.log(rng.uniform(1, 16, H)), dt_bias=0.1 * rng.standard_normal((H, D)),
        lower_bound=lb, scale=D ** -0.5,
        initial_state=None if zero_state else 0.3 * rng.standard_normal((N, H, D, D)),
        cu_seqlens=cu)
    return p


def run(oracle_mod, p, **over):
    args = dict(p)
    args.update(over)
    return oracle_mod.kda_oracle_fwd(**args)


# ---------------------------------------------------------------- unrolling
def unrolled(p, n, h):
    """Final state and outputs from explicit per-token transition matrices.

    With M_t = (I - b_t kh_t kh_t^T) diag(exp(a_t)) the recurrence is
    S_t = M_t S_{t-1} + b_t kh_t v_t^T, hence
    S_t = (M_t ... M_1) S_0 + sum_i (M_t ... M_{i+1}) b_i kh_i v_i^T,
    and o_t = scale * S_t^T qh_t.  Built here as dense products.
    """
    cu = p["cu_seqlens"]
    t0, t1 = cu[n], cu[n + 1]
    D = p["q"].shape[2]
    eps = 1e-6
    I = np.eye(D)
    Ms, Bs, outs = [], [], []
    S0 = np.zeros((D, D)) if p["initial_state"] is None else p["initial_state"][n, h]
    for t in range(t0, t1):
        qt, kt = p["q"][t, h], p["k"][t, h]
        kh = kt / math.sqrt(kt @ kt + eps)
        qh = qt / math.sqrt(qt @ qt + eps)
        x = math.exp(p["A_log"][h]) * (p["g"][t, h] + p["dt_bias"][h])
        a = p["lower_bound"] / (1.0 + np.exp(-x))
        b = 1.0 / (1.0 + math.exp(-p["beta"][t, h]))
        Ms.append((I - b * np.outer(kh, kh)) @ np.diag(np.exp(a)))
        Bs.append(b * np.outer(kh, p["v"][t, h]))
        # S_t from scratch as the explicit sum of products
        P = I.copy()
        S = np.zeros((D, D))
        for i in range(len(Ms) - 1, -1, -1):
            S += P @ Bs[i]
            P = P @ Ms[i]
        S += P @ S0
        outs.append(p["scale"] * S.T @ qh)
    return S if t1 > t0 else S0.copy(), np.array(outs)


@pytest.mark.parametrize("D", [4, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_unrolled_transition_products(oracle_mod, D, seed):
    rng = np.random.default_rng(seed)
    p = rand_problem(rng, None, 2, D, lengths=[12, 5, 9])
    out, fin = run(oracle_mod, p)
    cu = p["cu_seqlens"]
    for n in range(3):
        for h in range(2):
            S, o = unrolled(p, n, h)
            np.testing.assert_allclose(fin[n, h], S, rtol=0, atol=1e-12)
            np.testing.assert_allclose(out[cu[n]:cu[n + 1], h], o, rtol=0, atol=1e-12)


# ------------------------------------------------------------- chaining
@pytest.mark.parametrize("D,L", [(8, 40), (128, 150)])
def test_split_and_chain_reproduces_unsplit(oracle_mod, D, L):
    rng = np.random.default_rng(11)
    p = rand_problem(rng, None, 2, D, lengths=[L])
    out, fin = run(oracle_mod, p)
    for cut in [1, 7, L // 2, L - 1]:
        first = {k: (v[:cut] if k in ("q", "k", "v", "g", "beta") else v) for k, v in p.items()}
        first["cu_seqlens"] = np.array([0, cut], np.int32)
        o1, f1 = run(oracle_mod, first)
        second = {k: (v[cut:] if k in ("q", "k", "v", "g", "beta") else v) for k, v in p.items()}
        second["cu_seqlens"] = np.array([0, L - cut], np.int32)
        second["initial_state"] = f1
        o2, f2 = run(oracle_mod, second)
        np.testing.assert_allclose(np.concatenate([o1, o2]), out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(f2, fin, rtol=0, atol=1e-12)


# ------------------------------------------------------------- beta = 0
def test_beta_zero_only_decays(oracle_mod):
    """b = sigmoid(-BIG) = 0 exactly: S_t = diag(exp(Gamma_t)) S_0, no write."""
    rng = np.random.default_rng(3)
    D, L = 16, 30
    p = rand_problem(rng, None, 1, D, lengths=[L], lb=-0.7)
    p["beta"][:] = -BIG
    out, fin = run(oracle_mod, p)
    x = np.exp(p["A_log"][0]) * (p["g"][:, 0] + p["dt_bias"][0])
    a = p["lower_bound"] * 0.5 * (1.0 + np.tanh(0.5 * x))    # sigmoid via tanh
    Gam = np.cumsum(a, axis=0)
    S0 = p["initial_state"][0, 0]
    np.testing.assert_allclose(fin[0, 0], np.exp(Gam[-1])[:, None] * S0, rtol=1e-12, atol=1e-14)
    qh = p["q"][:, 0] / np.sqrt((p["q"][:, 0] ** 2).sum(1, keepdims=True) + 1e-6)
    expect = p["scale"] * np.einsum("td,dc->tc", qh * np.exp(Gam), S0)
    np.testing.assert_allclose(out[:, 0], expect, rtol=1e-11, atol=1e-13)


def test_state_rows_are_key_channels(oracle_mod):
    """Decay only key channel 0 (its gate logit -> +inf gives a = lb there,
    the others -> -inf give a = 0): only ROW 0 of the state shrinks."""
    rng = np.random.default_rng(4)
    D = 8
    p = rand_problem(rng, None, 1, D, lengths=[1], lb=-2.0)
    p["beta"][:] = -BIG
    p["dt_bias"][:] = 0.0
    p["g"][0, 0, :] = -BIG
    p["g"][0, 0, 0] = BIG
    _, fin = run(oracle_mod, p)
    S0 = p["initial_state"][0, 0]
    expect = S0.copy()
    expect[0, :] *= math.exp(-2.0)
    np.testing.assert_allclose(fin[0, 0], expect, rtol=1e-15, atol=0)


# ------------------------------------------------------------- gate values
@pytest.mark.parametrize("A_log,gsum,sig", [
    (0.0, 0.0, 0.5),                        # sigmoid(0) = 1/2
    (0.0, 1.0, 0.7310585786300049),         # sigmoid(1) = e/(1+e)
    (math.log(2.0), 1.0, 0.8807970779778823),  # exp(A_log)=2 -> sigmoid(2)
    (0.0, BIG, 1.0),                        # saturates at lower_bound
    (0.0, -BIG, 0.0),                       # no decay
])
def test_gate_known_values(oracle_mod, A_log, gsum, sig):
    """a = lb * sigmoid(exp(A_log) * (g + dt_bias)) at points with known sigmoid."""
    rng = np.random.default_rng(5)
    D, lb = 4, -3.0
    p = rand_problem(rng, None, 1, D, lengths=[1], lb=lb)
    p["beta"][:] = -BIG
    p["A_log"][:] = A_log
    p["dt_bias"][:] = 0.25
    p["g"][:] = gsum - 0.25
    _, fin = run(oracle_mod, p)
    S0 = p["initial_state"][0, 0]
    np.testing.assert_allclose(fin[0, 0], math.exp(lb * sig) * S0, rtol=1e-13, atol=0)


# ---------------------------------------------------- delta rule, exactness
def orthonormal_keys(rng, D, m, norm=1.0e3):
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    return norm * Qm[:, :m].T       # rows orthogonal, |row| = norm (eps negligible)


def test_orthonormal_writes_are_read_back_exactly(oracle_mod):
    """lb = 0 (no decay), b = 1 writes of orthogonal keys, then b = 0 reads
    with q = k_j and scale = 1 return v_j."""
    rng = np.random.default_rng(6)
    D, m = 16, 10
    keys = orthonormal_keys(rng, D, m)
    vals = rng.standard_normal((m, D))
    T = 2 * m
    p = rand_problem(rng, None, 1, D, lengths=[T], lb=0.0, zero_state=True)
    p["scale"] = 1.0
    p["k"][:m, 0] = keys
    p["v"][:m, 0] = vals
    p["beta"][:m, 0] = BIG
    order = rng.permutation(m)
    p["k"][m:, 0] = keys[order]              # read tokens: b = 0, any k
    p["q"][m:, 0] = keys[order]
    p["beta"][m:, 0] = -BIG
    out, fin = run(oracle_mod, p)
    np.testing.assert_allclose(out[m:, 0], vals[order], rtol=0, atol=1e-9)
    # the state is the sum of outer products kh_j v_j^T
    kh = keys / np.linalg.norm(keys, axis=1, keepdims=True)
    np.testing.assert_allclose(fin[0, 0], kh.T @ vals, rtol=0, atol=1e-9)


def test_overwrite_with_same_key(oracle_mod):
    """Writing (k, v1) then (k, v2) with b = 1 leaves S^T kh = v2."""
    rng = np.random.default_rng(7)
    D = 8
    p = rand_problem(rng, None, 1, D, lengths=[3], lb=0.0)
    p["scale"] = 1.0
    key = rng.standard_normal(D) * 100.0
    p["k"][:, 0] = key
    p["q"][:, 0] = key
    p["beta"][:2, 0] = BIG
    p["beta"][2, 0] = -BIG
    out, fin = run(oracle_mod, p)
    kh = key / np.linalg.norm(key)
    np.testing.assert_allclose(fin[0, 0].T @ kh, p["v"][1, 0], rtol=0, atol=1e-9)
    np.testing.assert_allclose(out[2, 0], p["v"][1, 0], rtol=0, atol=1e-9)
    np.testing.assert_allclose(out[1, 0], p["v"][1, 0], rtol=0, atol=1e-9)  # read after write


def test_single_token_from_zero_state(oracle_mod):
    """o = scale * b * (qh . kh) v and S = b kh v^T (the read follows the write)."""
    rng = np.random.default_rng(8)
    D = 32
    p = rand_problem(rng, None, 3, D, lengths=[1], zero_state=True)
    out, fin = run(oracle_mod, p)
    for h in range(3):
        q, k, v = p["q"][0, h], p["k"][0, h], p["v"][0, h]
        qh, kh = q / np.linalg.norm(q), k / np.linalg.norm(k)
        b = 1.0 / (1.0 + math.exp(-p["beta"][0, h]))
        np.testing.assert_allclose(out[0, h], p["scale"] * b * (qh @ kh) * v, rtol=1e-5, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], b * np.outer(kh, v), rtol=1e-5, atol=1e-12)


# ------------------------------------------------------------- invariants
def test_normalisation_and_scale(oracle_mod):
    rng = np.random.default_rng(9)
    D = 16
    p = rand_problem(rng, None, 2, D, lengths=[20])
    out, fin = run(oracle_mod, p)
    # eps = 1e-6 against |k|^2 ~ 16 perturbs the unit vectors by ~3e-8
    out2, fin2 = run(oracle_mod, p, q=p["q"] * 7.5, k=p["k"] * 3.0)
    np.testing.assert_allclose(out2, out, rtol=0, atol=2e-7)
    np.testing.assert_allclose(fin2, fin, rtol=0, atol=2e-7)
    out3, fin3 = run(oracle_mod, p, scale=2.0 * p["scale"])
    np.testing.assert_allclose(out3, 2.0 * out, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin3, fin, rtol=0, atol=0)
    q0 = p["q"].copy()
    q0[5] = 0.0
    out4, _ = run(oracle_mod, p, q=q0)
    assert np.all(out4[5] == 0.0)


def test_packing_permutation_and_heads(oracle_mod):
    """Each (sequence, head) pair is independent of the others and of order."""
    rng = np.random.default_rng(10)
    D = 8
    lens = [5, 0, 13, 1, 9]
    p = rand_problem(rng, None, 3, D, lengths=lens)
    out, fin = run(oracle_mod, p)
    cu = p["cu_seqlens"]
    perm = [3, 0, 4, 2, 1]
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in perm]).astype(int)
    q = {k: p[k][rows] for k in ("q", "k", "v", "g", "beta")}
    plens = [lens[n] for n in perm]
    pcu = np.concatenate([[0], np.cumsum(plens)]).astype(np.int32)
    outp, finp = run(oracle_mod, p, **q, cu_seqlens=pcu,
                     initial_state=p["initial_state"][perm])
    np.testing.assert_array_equal(outp, out[rows])
    np.testing.assert_array_equal(finp, fin[perm])
    # one head alone gives the same as inside the batch
    h = 2
    one = {k: p[k][:, h:h + 1] for k in ("q", "k", "v", "g", "beta")}
    o1, f1 = run(oracle_mod, p, **one, A_log=p["A_log"][h:h + 1],
                 dt_bias=p["dt_bias"][h:h + 1], initial_state=p["initial_state"][:, h:h + 1])
    np.testing.assert_array_equal(o1[:, 0], out[:, h])
    np.testing.assert_array_equal(f1[:, 0], fin[:, h])
    # the empty sequence passes its initial state through
    np.testing.assert_array_equal(fin[1], p["initial_state"][1])


def test_tokens_past_last_sequence_untouched(oracle_mod):
    rng = np.random.default_rng(12)
    D = 8
    p = rand_problem(rng, None, 1, D, lengths=[6])
    for key in ("q", "k", "v", "g"):
        p[key] = np.concatenate([p[key], rng.standard_normal((4, 1, D))])
    p["beta"] = np.concatenate([p["beta"], rng.standard_normal((4, 1))])
    out, _ = run(oracle_mod, p)
    assert np.all(out[6:] == 0.0)


def test_rejects_bad_cu_seqlens(oracle_mod):
    rng = np.random.default_rng(13)
    p = rand_problem(rng, None, 1, 4, lengths=[3, 3])
    with pytest.raises(ValueError):
        run(oracle_mod, p, cu_seqlens=np.array([0, 4, 3], np.int32))
    with pytest.raises(ValueError):
        run(oracle_mod, p, cu_seqlens=np.array([1, 3, 6], np.int32))
    with pytest.raises(ValueError):
        run(oracle_mod, p, cu_seqlens=np.array([0, 3, 7], np.int32))
