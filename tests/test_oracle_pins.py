"""Pins for the double-precision oracle, independent of the oracle itself.

Each check compares the oracle with something the pages or the mathematics
fix: the printed prefix-sum and Blelloch examples, the LTI convolution
written out by brute force, the chunk-carry identity, the cumulative-product
closed form, every bracketing of the associative operator, and special cases
with closed forms.  ``test_every_planted_mistake_is_caught`` runs the pin set
against the oracle with deliberate slips planted in it (a dropped term, a
sign, an index, an operand swap) and requires each slip to fail some pin.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- pscan pins

def test_prefix_sum_golden():
    g = read_golden("prefix_sum.txt")
    x = np.array(g["input"][0])
    want = np.array(g["output"][0])
    ones = np.ones_like(x)
    got = oracle.pscan_seq(ones[None], x[None])[0]
    assert np.array_equal(got, want)
    got_b = oracle.pscan_blelloch(ones, x)
    assert np.array_equal(got_b, want)


def test_blelloch_upsweep_trace_golden():
    g = read_golden("blelloch_upsweep.txt")
    x = np.array(g["input"][0])
    levels = np.array(g["level"])
    h, (ta, tb) = oracle.pscan_blelloch(np.ones_like(x), x, trace=True)
    assert ta.shape[0] == 3 and tb.shape == (3, 8)
    assert np.array_equal(tb, levels)
    assert np.all(ta == 1.0)
    # the inclusive result, by brute force: each output is the sum of its prefix
    brute = np.array([sum(x[: i + 1]) for i in range(len(x))])
    assert np.array_equal(h, brute)
    assert list(brute) == [1, 3, 6, 10, 15, 21, 28, 36]


def _pscan_brute(a, b, h0):
    """h_k = (prod_{j<=k} a_j) h0 + sum_{i<=k} (prod_{i<j<=k} a_j) b_i, by explicit
    products (O(n^2)); no recurrence."""
    n = len(a)
    out = np.zeros(n)
    for k in range(n):
        acc = np.prod(a[: k + 1]) * h0
        for i in range(k + 1):
            acc += np.prod(a[i + 1: k + 1]) * b[i]
        out[k] = acc
    return out


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 13, 37])
def test_pscan_seq_and_blelloch_vs_explicit_products(n):
    r = _rng(100 + n)
    a = r.uniform(-1.3, 1.3, n)   # signs and |a| > 1: the operator is not commutative here
    b = r.normal(size=n)
    h0 = float(r.normal())
    brute = _pscan_brute(a, b, h0)
    seq = oracle.pscan_seq(a[None], b[None], np.array([h0]))[0]
    ble = oracle.pscan_blelloch(a, b, h0)
    np.testing.assert_allclose(seq, brute, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ble, brute, rtol=1e-12, atol=1e-12)


def test_pscan_cumulative_product_closed_form():
    """x_k = A'_k x_0 + sum_i (A'_k / A'_i) B_i u_i with A'_k = prod_{i<=k} A_i
    ("图解Blelloch并行扫描", section 3.1), for A in [0.5, 1] where the division is safe."""
    r = _rng(7)
    n = 40
    a = r.uniform(0.5, 1.0, n)
    bu = r.normal(size=n)
    x0 = 0.75
    Ap = np.cumprod(a)
    closed = np.array([Ap[k] * x0 + sum(Ap[k] / Ap[i] * bu[i] for i in range(k + 1))
                       for k in range(n)])
    got = oracle.pscan_seq(a[None], bu[None], np.array([x0]))[0]
    np.testing.assert_allclose(got, closed, rtol=1e-12)


def _bracketings(items):
    """Every full binary tree over the ordered list, as a combined (a, b) pair."""
    if len(items) == 1:
        yield items[0]
        return
    for cut in range(1, len(items)):
        for left in _bracketings(items[:cut]):
            for right in _bracketings(items[cut:]):
                a1, b1 = left
                a2, b2 = right
                yield (a2 * a1, a2 * b1 + b2)


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6, 7, 8])
def test_every_bracketing_matches_the_oracle_fold_dyadic(n):
    """Associativity of (a1,b1)o(a2,b2) = (a2 a1, a2 b1 + b2): every bracketing of n
    pairs gives the oracle's sequential result bit for bit on dyadic inputs."""
    r = _rng(200 + n)
    a = r.choice([0.5, -0.5, 0.25, -0.25, 1.0], size=n)
    b = r.integers(-8, 9, size=n).astype(np.float64)
    seq = oracle.pscan_seq(a[None], b[None])[0][-1]
    ble = oracle.pscan_blelloch(a, b)[-1]
    count = 0
    for A_, B_ in _bracketings(list(zip(a, b))):
        assert B_ == seq and B_ == ble
        assert A_ == np.prod(a)
        count += 1
    assert count == math.comb(2 * (n - 1), n - 1) // n  # Catalan(n-1) trees


@pytest.mark.parametrize("n", [3, 6, 8])
def test_every_bracketing_matches_the_oracle_fold_random(n):
    r = _rng(300 + n)
    a = r.uniform(-1.2, 1.2, n)
    b = r.normal(size=n)
    seq = oracle.pscan_seq(a[None], b[None])[0][-1]
    for _, B_ in _bracketings(list(zip(a, b))):
        assert abs(B_ - seq) <= 1e-15 * max(1.0, abs(seq)) * 8


# ----------------------------------------------------- selective-scan pins
# Each pin takes a callable sscan(u, delta, A, B, C, D, h0) -> (y, hT) and
# returns None when it holds, else a message.


def _rand_problem(seed, batch=2, dim=3, L=17, N=4, h0=True, D=True):
    r = _rng(seed)
    u = r.normal(size=(batch, dim, L))
    delta = np.log1p(np.exp(r.normal(-1.0, 0.7, size=(batch, dim, L))))
    A = -r.uniform(0.2, 3.0, size=(dim, N))
    B = r.normal(size=(batch, N, L))
    C = r.normal(size=(batch, N, L))
    Dv = r.normal(size=dim) if D else None
    h0v = r.normal(size=(batch, dim, N)) * 0.5 if h0 else None
    return u, delta, A, B, C, Dv, h0v


def pin_lti_convolution(sscan):
    """Constant delta, B, C over t: y_k = sum_{i<=k} C Abar^i Bbar u_{k-i}
    + C Abar^{k+1} h0 + D u_k, with Abar = exp(delta A), Bbar = delta B
    ("Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战", section 1.3), by brute-force convolution."""
    r = _rng(11)
    batch, dim, L, N = 2, 3, 40, 5
    dval = r.uniform(0.05, 0.6, size=(batch, dim))
    delta = np.repeat(dval[:, :, None], L, axis=2)
    u = r.normal(size=(batch, dim, L))
    A = -r.uniform(0.1, 2.0, size=(dim, N))
    Bc = r.normal(size=(batch, N))
    Cc = r.normal(size=(batch, N))
    B = np.repeat(Bc[:, :, None], L, axis=2)
    C = np.repeat(Cc[:, :, None], L, axis=2)
    D = r.normal(size=dim)
    h0 = r.normal(size=(batch, dim, N))
    y, hT = sscan(u, delta, A, B, C, D, h0)
    for b in range(batch):
        for d in range(dim):
            Ab = np.exp(dval[b, d] * A[d])            # [N]
            Bb = dval[b, d] * Bc[b]                   # [N]
            kern = np.array([np.sum(Cc[b] * Ab ** i * Bb) for i in range(L)])
            for k in range(L):
                want = sum(kern[i] * u[b, d, k - i] for i in range(k + 1))
                want += np.sum(Cc[b] * Ab ** (k + 1) * h0[b, d]) + D[d] * u[b, d, k]
                if abs(y[b, d, k] - want) > 1e-12 * (1 + abs(want)):
                    return f"LTI y[{b},{d},{k}] {y[b, d, k]} != {want}"
            hw = Ab ** L * h0[b, d] + sum(Ab ** (L - 1 - i) * Bb * u[b, d, i] for i in range(L))
            if np.max(np.abs(hT[b, d] - hw)) > 1e-12 * (1 + np.max(np.abs(hw))):
                return "LTI final state"
    return None


def pin_chunk_identity_page_example(sscan):
    """The chunk-carry identity with the page's diagonal A-bar and chunk 3:
    h_{3k} = Abar^3 h_{3(k-1)} + sum_{i=0}^{2} Abar^{2-i} Bbar x_{3(k-1)+i+1}
    ("为什么Mamba的“并行扫描”不是真并行 (mhpq.cn/news/1057127)", section 3; the index is read as in the
    page's own simulation, h3 = A^3 h0 + A^2 Bx1 + A Bx2 + Bx3)."""
    g = read_golden("chunk_carry_diag.txt")
    abar = np.array(g["abar"][0])
    ck = int(g["chunk"][0][0])
    N = abar.size
    r = _rng(12)
    L = 4 * ck
    u = r.normal(size=(1, 1, L))
    delta = np.ones((1, 1, L))                 # delta = 1 so that exp(delta A) = abar
    A = np.log(abar)[None, :]
    Bv = r.normal(size=(1, N, L))
    C = np.zeros((1, N, L))
    h0 = r.normal(size=(1, 1, N))
    bx = Bv[0] * u[0, 0][None, :]              # Bbar x_t, [N, L]  (delta = 1)
    h = h0[0, 0].copy()
    for k in range(1, L // ck + 1):
        s = (k - 1) * ck
        h = abar ** ck * h + sum(abar ** (ck - 1 - i) * bx[:, s + i] for i in range(ck))
        _, hT = sscan(u[:, :, :k * ck], delta[:, :, :k * ck], A,
                      Bv[:, :, :k * ck], C[:, :, :k * ck], None, h0)
        if np.max(np.abs(hT[0, 0] - h)) > 1e-12 * (1 + np.max(np.abs(h))):
            return f"chunk identity at h_{k * ck}"
    return None


def pin_chunk_identity_selective(sscan):
    """Selective form of the chunk carry: over a chunk [s, e), the diagonal power
    becomes prod_t exp(delta_t A) = exp(A sum_t delta_t), and the chunk's own
    contribution is sum_t exp(A sum_{j>t} delta_j) delta_t u_t B_t.  Chained
    over chunks of 1, 3, 7 and 64 steps it must reproduce the end state."""
    u, delta, A, B, C, D, h0 = _rand_problem(13, batch=1, dim=2, L=150, N=3)
    _, hT = sscan(u, delta, A, B, C, D, h0)
    for ck in (1, 3, 7, 64):
        for d in range(2):
            h = h0[0, d].copy()
            for s in range(0, 150, ck):
                e = min(s + ck, 150)
                dl = delta[0, d, s:e]
                h = np.exp(A[d] * dl.sum()) * h + sum(
                    np.exp(A[d] * dl[t + 1:].sum()) * dl[t] * u[0, d, s + t] * B[0, :, s + t]
                    for t in range(e - s))
            if np.max(np.abs(hT[0, d] - h)) > 1e-11 * (1 + np.max(np.abs(h))):
                return f"selective chunk identity, chunk {ck}"
    return None


def pin_A_zero_is_prefix_sum(sscan):
    """A = 0 gives Abar = 1, so h_t = h0 + sum_{s<=t} delta_s u_s B_s, a plain
    prefix sum (cumsum), and y_t = C_t . h_t + D u_t."""
    u, delta, _, B, C, D, h0 = _rand_problem(14, N=3)
    A = np.zeros((u.shape[1], 3))
    y, hT = sscan(u, delta, A, B, C, D, h0)
    for b in range(u.shape[0]):
        for d in range(u.shape[1]):
            x = delta[b, d][None, :] * u[b, d][None, :] * B[b]       # [N, L]
            h = h0[b, d][:, None] + np.cumsum(x, axis=1)
            want = np.sum(C[b] * h, axis=0) + D[d] * u[b, d]
            if np.max(np.abs(y[b, d] - want)) > 1e-12 * (1 + np.max(np.abs(want))):
                return "A = 0 prefix sum"
            if np.max(np.abs(hT[b, d] - h[:, -1])) > 1e-12 * (1 + np.max(np.abs(h))):
                return "A = 0 final state"
    return None


def pin_instant_decay(sscan):
    """delta*A -> -inf gives Abar = 0: h_t = delta_t u_t B_t and
    y_t = delta_t u_t (C_t . B_t) + D u_t, whatever h0 was."""
    u, delta, _, B, C, D, h0 = _rand_problem(15, N=4)
    A = np.full((u.shape[1], 4), -1e300)
    y, hT = sscan(u, delta, A, B, C, D, h0)
    for b in range(u.shape[0]):
        for d in range(u.shape[1]):
            du = delta[b, d] * u[b, d]
            want = du * np.sum(C[b] * B[b], axis=0) + D[d] * u[b, d]
            if np.max(np.abs(y[b, d] - want)) > 1e-12 * (1 + np.max(np.abs(want))):
                return "instant decay output"
            if np.max(np.abs(hT[b, d] - du[-1] * B[b, :, -1])) > 1e-12:
                return "instant decay final state"
    return None


def pin_C_zero_gives_skip_only(sscan):
    """C = 0 leaves only the skip term: y = D u exactly (bit for bit)."""
    u, delta, A, B, _, D, h0 = _rand_problem(16, N=4)
    C = np.zeros_like(B)
    y, _ = sscan(u, delta, A, B, C, D, h0)
    want = D[None, :, None] * u
    return None if np.array_equal(y, want) else "C = 0 skip term"


def pin_single_step(sscan):
    """L = 1: y_0 = sum_n C_0 (exp(delta_0 A) h0 + delta_0 B_0 u_0) + D u_0."""
    u, delta, A, B, C, D, h0 = _rand_problem(17, L=1, N=5)
    y, hT = sscan(u, delta, A, B, C, D, h0)
    for b in range(u.shape[0]):
        for d in range(u.shape[1]):
            h1 = np.exp(delta[b, d, 0] * A[d]) * h0[b, d] + delta[b, d, 0] * B[b, :, 0] * u[b, d, 0]
            want = np.sum(C[b, :, 0] * h1) + D[d] * u[b, d, 0]
            if abs(y[b, d, 0] - want) > 1e-13 * (1 + abs(want)):
                return "single step output"
            if np.max(np.abs(hT[b, d] - h1)) > 1e-13 * (1 + np.max(np.abs(h1))):
                return "single step state"
    return None


def pin_state_passing(sscan):
    """One call over L equals two calls over [0, m) and [m, L) that pass the
    first call's final state as the second call's h0."""
    u, delta, A, B, C, D, h0 = _rand_problem(18, L=29, N=3)
    y, hT = sscan(u, delta, A, B, C, D, h0)
    m = 11
    y1, h1 = sscan(u[..., :m], delta[..., :m], A, B[..., :m], C[..., :m], D, h0)
    y2, h2 = sscan(u[..., m:], delta[..., m:], A, B[..., m:], C[..., m:], D, h1)
    if np.max(np.abs(np.concatenate([y1, y2], axis=2) - y)) > 1e-12 * (1 + np.max(np.abs(y))):
        return "state passing output"
    if np.max(np.abs(h2 - hT)) > 1e-12 * (1 + np.max(np.abs(hT))):
        return "state passing final state"
    return None


PINS = [pin_lti_convolution, pin_chunk_identity_page_example,
        pin_chunk_identity_selective, pin_A_zero_is_prefix_sum, pin_instant_decay,
        pin_C_zero_gives_skip_only, pin_single_step, pin_state_passing]


def _oracle_callable(mutation=0):
    def f(u, delta, A, B, C, D, h0):
        return oracle.sscan_fwd(u, delta, A, B, C, D, h0, mutation=mutation)
    return f


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    msg = pin(_oracle_callable())
    assert msg is None, msg


def test_every_planted_mistake_is_caught():
    for m in BASE_MUTATIONS:
        f = _oracle_callable(m)
        failed = [p.__name__ for p in PINS if p(f) is not None]
        assert failed, f"planted mistake {m} passed every pin"


# ------------------------------------------- pins of the scan's options
# Each takes full(u, delta, A, B, C, D, z, delta_bias, h0, softplus, zoh)
# -> (y, hT) and returns None when it holds, else a message.

BASE_MUTATIONS = range(1, 9)     # planted in the plain scan
OPTION_MUTATIONS = range(9, 14)  # planted in softplus / gate / zero-order hold


def pin_softplus_inverse(full):
    """delta_softplus: softplus(r + bias) = k exactly when r = log(e^k - 1) - bias
    ("CUDA 内核优化实战" section 7.1 applies softplus inside the op; section 2.2
    defines delta as softplus of a projection, whose bias is delta_bias)."""
    u, _, A, B, C, D, h0 = _rand_problem(31)
    r = _rng(32)
    k = r.uniform(0.01, 3.0, size=u.shape)
    bias = r.normal(size=u.shape[1])
    raw = np.log(np.expm1(k)) - bias[None, :, None]
    y_ref, h_ref = oracle.sscan_fwd(u, k, A, B, C, D, h0)
    y, hT = full(u, raw, A, B, C, D, None, bias, h0, True, False)
    if np.max(np.abs(y - y_ref)) > 1e-12 * (1 + np.max(np.abs(y_ref))):
        return "softplus(delta + bias) output"
    if np.max(np.abs(hT - h_ref)) > 1e-12 * (1 + np.max(np.abs(h_ref))):
        return "softplus(delta + bias) final state"
    # without softplus the bias alone shifts delta
    y, _ = full(u, k - bias[None, :, None], A, B, C, D, None, bias, h0, False, False)
    if np.max(np.abs(y - y_ref)) > 1e-12 * (1 + np.max(np.abs(y_ref))):
        return "delta + bias output"
    return None


def pin_gate_special_values(full):
    """z-gate out = (y + D u) * z * sigmoid(z) at points where silu has a closed
    form: silu(0) = 0, silu(40) = 40 to double precision, silu(+-ln 3) =
    +-ln 3 * (3/4 or 1/4)."""
    u, delta, A, B, C, D, h0 = _rand_problem(33)
    y0, h0ref = oracle.sscan_fwd(u, delta, A, B, C, D, h0)
    pick = _rng(34).integers(0, 5, size=u.shape)
    ln3 = np.log(3.0)
    zvals = np.array([0.0, 40.0, ln3, -ln3, 40.0])
    gate = np.array([0.0, 40.0, 0.75 * ln3, -0.25 * ln3, 40.0])
    z = zvals[pick]
    y, hT = full(u, delta, A, B, C, D, z, None, h0, False, False)
    if np.max(np.abs(y - y0 * gate[pick])) > 1e-12 * (1 + np.max(np.abs(y0 * 40))):
        return "gated output"
    if np.max(np.abs(hT - h0ref)) > 0:
        return "the gate must not touch the state"
    return None


def _zoh_by_ode(u, delta, A, B, C, D, h0, substeps=400):
    """Integrate dh/dt = A h + B_t u_t over each step's duration delta_t with the
    input held (RK4, many substeps) -- the zero-order hold by its definition,
    independent of the closed form."""
    batch, dim, L = u.shape
    N = A.shape[1]
    y = np.zeros((batch, dim, L))
    hT = np.zeros((batch, dim, N))
    for b in range(batch):
        for d in range(dim):
            h = h0[b, d].copy() if h0 is not None else np.zeros(N)
            a = A[d]
            for t in range(L):
                f = B[b, :, t] * u[b, d, t]
                dt = delta[b, d, t] / substeps
                for _ in range(substeps):
                    k1 = a * h + f
                    k2 = a * (h + 0.5 * dt * k1) + f
                    k3 = a * (h + 0.5 * dt * k2) + f
                    k4 = a * (h + dt * k3) + f
                    h = h + dt / 6.0 * (k1 + 2 * k2 + 2 * k3 + k4)
                y[b, d, t] = C[b, :, t] @ h + (D[d] * u[b, d, t] if D is not None else 0.0)
            hT[b, d] = h
    return y, hT


def pin_zoh_matches_ode(full):
    """ZOH B-bar ("CUDA 内核优化实战" section 1.2): the discrete step equals the
    exact solution of the continuous system over a step with the input held."""
    u, delta, A, B, C, D, h0 = _rand_problem(35, batch=1, dim=2, L=9, N=3)
    y_ode, h_ode = _zoh_by_ode(u, delta, A, B, C, D, h0)
    y, hT = full(u, delta, A, B, C, D, None, None, h0, False, True)
    if np.max(np.abs(y - y_ode)) > 1e-9 * (1 + np.max(np.abs(y_ode))):
        return "zoh output vs the integrated ODE"
    if np.max(np.abs(hT - h_ode)) > 1e-9 * (1 + np.max(np.abs(h_ode))):
        return "zoh final state vs the integrated ODE"
    return None


def pin_zoh_small_A_is_euler(full):
    """As A -> 0 the ZOH B-bar tends to delta*B (A = 0 exactly: equal)."""
    u, delta, A, B, C, D, h0 = _rand_problem(36)
    A0 = np.zeros_like(A)
    y_e, h_e = oracle.sscan_fwd(u, delta, A0, B, C, D, h0)
    y_z, h_z = full(u, delta, A0, B, C, D, None, None, h0, False, True)
    if np.max(np.abs(y_z - y_e)) > 1e-13 * (1 + np.max(np.abs(y_e))):
        return "zoh with A = 0"
    y_e, _ = oracle.sscan_fwd(u, delta, A0 - 1e-9, B, C, D, h0)
    y_z, _ = full(u, delta, A0 - 1e-9, B, C, D, None, None, h0, False, True)
    if np.max(np.abs(y_z - y_e)) > 1e-7 * (1 + np.max(np.abs(y_e))):
        return "zoh with A = -1e-9"
    return None


OPTION_PINS = [pin_softplus_inverse, pin_gate_special_values, pin_zoh_matches_ode,
               pin_zoh_small_A_is_euler]


def _full_callable(mutation=0):
    def f(u, delta, A, B, C, D, z, bias, h0, softplus, zoh):
        return oracle.sscan_fwd_full(u, delta, A, B, C, D, z, bias, h0, delta_softplus=softplus,
                                     zoh=zoh, mutation=mutation)
    return f


@pytest.mark.parametrize("pin", OPTION_PINS, ids=lambda p: p.__name__)
def test_oracle_option_pin(pin):
    msg = pin(_full_callable())
    assert msg is None, msg


def test_every_planted_option_mistake_is_caught():
    assert oracle.mutation_count() == OPTION_MUTATIONS[-1] + 1
    for m in OPTION_MUTATIONS:
        f = _full_callable(m)
        failed = [p.__name__ for p in OPTION_PINS if p(f) is not None]
        assert failed, f"planted option mistake {m} passed every pin"


def test_the_copy_carrying_the_planted_mistakes_equals_the_definition():
    """The planted-mistake tests run on a copy of the definition, so that the
    definition itself carries no mistake switches; with no mistake planted
    (code 100) that copy computes exactly what the definition computes, with
    every option on and off, threaded or not."""
    u, delta, A, B, C, D, h0 = _rand_problem(41)
    r = _rng(42)
    z = r.normal(size=u.shape)
    bias = r.normal(size=A.shape[0]) * 0.3
    A = A.copy()
    A[0, 1] = 0.0  # the zero-order hold's A = 0 branch
    for softplus in (False, True):
        for zoh in (False, True):
            for gate in (None, z):
                for nth in (1, 3):
                    ref = oracle.sscan_fwd_full(u, delta, A, B, C, D, gate, bias, h0,
                                                delta_softplus=softplus, zoh=zoh, nthreads=nth)
                    cp = oracle.sscan_fwd_full(u, delta, A, B, C, D, gate, bias, h0,
                                               delta_softplus=softplus, zoh=zoh, nthreads=nth,
                                               mutation=100)
                    assert np.array_equal(ref[0], cp[0]) and np.array_equal(ref[1], cp[1])


def test_options_off_is_the_plain_scan():
    u, delta, A, B, C, D, h0 = _rand_problem(37)
    y0, h0r = oracle.sscan_fwd(u, delta, A, B, C, D, h0)
    y1, h1 = oracle.sscan_fwd_full(u, delta, A, B, C, D, None, None, h0)
    assert np.array_equal(y0, y1) and np.array_equal(h0r, h1)


# ------------------------------------------------- pins of the gradients
# The backward oracle is pinned to central finite differences of the forward
# oracle (itself pinned above) on the loss L = sum dy*y + sum dhT*final_state.


def _fd_gradients(u, delta, A, B, C, D, h0, dy, dhT, eps=1e-6):
    args = {"u": u, "delta": delta, "A": A, "B": B, "C": C, "D": D, "h0": h0}

    def loss(a):
        y, hT = oracle.sscan_fwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["h0"])
        return float(np.sum(dy * y) + np.sum(dhT * hT))

    grads = {}
    for name, x in args.items():
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            e = eps * max(1.0, abs(x[idx]))
            xp = x.copy()
            xp[idx] += e
            xm = x.copy()
            xm[idx] -= e
            gx[idx] = (loss({**args, name: xp}) - loss({**args, name: xm})) / (2 * e)
        grads[name] = gx
    return grads


def pin_bwd_finite_differences(bwd):
    """Every gradient of the scan against central finite differences."""
    u, delta, A, B, C, D, h0 = _rand_problem(41, batch=2, dim=2, L=6, N=3)
    r = _rng(42)
    dy = r.normal(size=u.shape)
    dhT = r.normal(size=h0.shape)
    fd = _fd_gradients(u, delta, A, B, C, D, h0, dy, dhT)
    g = bwd(u, delta, A, B, C, D, h0, dy, dhT)
    pairs = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "h0": "dh0"}
    for x, gname in pairs.items():
        err = np.max(np.abs(g[gname] - fd[x]) / (1 + np.abs(fd[x])))
        if err > 1e-6:
            return f"{gname} vs finite differences: {err:.2e}"
    return None


def pin_bwd_no_upstream_is_zero(bwd):
    """dy = 0 and dhT = 0 give zero gradients everywhere."""
    u, delta, A, B, C, D, h0 = _rand_problem(43)
    g = bwd(u, delta, A, B, C, D, h0, np.zeros_like(u), np.zeros_like(h0))
    if any(np.any(v != 0) for v in g.values() if v is not None):
        return "nonzero gradient without upstream gradient"
    return None


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_no_upstream_is_zero]


def _bwd_callable(mutation=0):
    def f(u, delta, A, B, C, D, h0, dy, dhT):
        return oracle.sscan_bwd(u, delta, A, B, C, D, h0, dy, dhT, mutation=mutation)
    return f


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
def test_oracle_bwd_pin(pin):
    msg = pin(_bwd_callable())
    assert msg is None, msg


def test_every_planted_bwd_mistake_is_caught():
    for m in range(1, oracle.bwd_mutation_count()):
        failed = [p.__name__ for p in BWD_PINS if p(_bwd_callable(m)) is not None]
        assert failed, f"planted backward mistake {m} passed every pin"


def test_threaded_oracle_equals_single_thread():
    u, delta, A, B, C, D, h0 = _rand_problem(19, batch=3, dim=5, L=33, N=4)
    y1, h1 = oracle.sscan_fwd(u, delta, A, B, C, D, h0, nthreads=1)
    y4, h4 = oracle.sscan_fwd(u, delta, A, B, C, D, h0, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(h1, h4)


def test_channel_sample_equals_full_problem():
    u, delta, A, B, C, D, h0 = _rand_problem(20, batch=2, dim=4, L=21, N=3)
    y, hT = oracle.sscan_fwd(u, delta, A, B, C, D, h0)
    chans = [(0, 3), (1, 0), (1, 2)]
    ys, hs = oracle.sscan_fwd_channels(u, delta, A, B, C, D, h0, chans)
    for i, (b, d) in enumerate(chans):
        assert np.array_equal(ys[i], y[b, d]) and np.array_equal(hs[i], hT[b, d])


def test_oracle_empty_and_degenerate_sizes():
    y, hT = oracle.sscan_fwd(np.zeros((1, 2, 0)), np.zeros((1, 2, 0)),
                             np.zeros((2, 3)), np.zeros((1, 3, 0)), np.zeros((1, 3, 0)))
    assert y.shape == (1, 2, 0) and np.array_equal(hT, np.zeros((1, 2, 3)))
    # N = 0: no state, y = D u
    u = _rng(1).normal(size=(1, 2, 5))
    D = np.array([2.0, -1.0])
    y, _ = oracle.sscan_fwd(u, np.ones_like(u), np.zeros((2, 0)), np.zeros((1, 0, 5)),
                            np.zeros((1, 0, 5)), D)
    assert np.array_equal(y, D[None, :, None] * u)
