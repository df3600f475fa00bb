"""Pins of the Mamba-2 recurrence oracle against things other than itself: closed forms
(no decay, full decay, an impulse response), the state-space-duality matrix form
written independently, and state carry-over across split calls."""
import numpy as np

from oracle import ssd


def _inputs(rng, T, H, P, N, G):
    x = rng.standard_normal((T, H, P))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    loga = -np.abs(rng.standard_normal((T, H))) * 0.3
    return x, B, C, loga


def test_no_decay_is_a_running_sum():
    rng = np.random.default_rng(1)
    T, H, P, N = 9, 2, 3, 4
    x, B, C, _ = _inputs(rng, T, H, P, N, 1)
    y, _ = ssd.ssd_scan(x, B, C, np.zeros((T, H)))
    for t in range(T):
        for h in range(H):
            want = sum((C[t, 0] @ B[j, 0]) * x[j, h] for j in range(t + 1))
            assert np.allclose(y[t, h], want, rtol=1e-12, atol=1e-12)


def test_full_decay_keeps_only_the_current_token():
    rng = np.random.default_rng(2)
    T, H, P, N = 7, 3, 2, 5
    x, B, C, _ = _inputs(rng, T, H, P, N, 1)
    y, _ = ssd.ssd_scan(x, B, C, np.full((T, H), -np.inf))
    for t in range(T):
        assert np.allclose(y[t], (C[t, 0] @ B[t, 0]) * x[t], rtol=1e-12)


def test_impulse_response_decays_geometrically():
    T, H, P, N = 12, 1, 2, 3
    x = np.zeros((T, H, P))
    x[3, 0] = [1.0, -2.0]
    B = np.ones((T, 1, N))
    C = np.ones((T, 1, N)) * 0.5
    loga = np.full((T, H), np.log(0.9))
    y, _ = ssd.ssd_scan(x, B, C, loga)
    for t in range(T):
        want = 0.0 if t < 3 else 0.9 ** (t - 3) * 0.5 * N
        assert np.allclose(y[t, 0], want * np.array([1.0, -2.0]), rtol=1e-12, atol=1e-15)


def test_matches_duality_matrix_form_with_groups():
    """y_t = sum_{s <= t} exp(sum_{r = s+1..t} loga_r) (C_t . B_s) x_s: the masked
    'attention' form of the same recurrence, computed per head with matrices."""
    rng = np.random.default_rng(3)
    T, H, P, N, G = 40, 4, 6, 8, 2
    x, B, C, loga = _inputs(rng, T, H, P, N, G)
    y, _ = ssd.ssd_scan(x, B, C, loga, n_groups=G)
    for h in range(H):
        g = h // (H // G)
        cum = np.cumsum(loga[:, h])
        L = np.exp(cum[:, None] - cum[None, :]) * np.tril(np.ones((T, T)))
        M = L * (C[:, g] @ B[:, g].T)
        assert np.allclose(y[:, h], M @ x[:, h], rtol=1e-10, atol=1e-10)


def test_split_calls_carry_the_state():
    rng = np.random.default_rng(4)
    T, H, P, N = 30, 2, 4, 6
    x, B, C, loga = _inputs(rng, T, H, P, N, 1)
    y, st = ssd.ssd_scan(x, B, C, loga)
    y1, s1 = ssd.ssd_scan(x[:11], B[:11], C[:11], loga[:11])
    y2, s2 = ssd.ssd_scan(x[11:], B[11:], C[11:], loga[11:], state0=s1)
    assert np.allclose(np.concatenate([y1, y2]), y, rtol=1e-12, atol=1e-12)
    assert np.allclose(s2, st, rtol=1e-12, atol=1e-12)
