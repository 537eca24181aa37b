"""Library pipeline model and auto-configurator (host code, no GPU) against
the oracle's restatement of Eq. 5 and a brute-force search of Eqs. 8-10."""
import itertools
import math

import numpy as np
import pytest

import oracle
from routed_expert_ffn_topk_gb300 import build as build_mod


@pytest.fixture(scope="module")
def es():
    build_mod.build()
    from routed_expert_ffn_topk_gb300 import estream
    return estream


def test_maxplus_matches_oracle(es):
    rng = np.random.default_rng(11)
    for K, q, b in itertools.product((1, 3, 8, 25), (1, 2, 4), (1, 2, 3, 7)):
        L = rng.uniform(0.0, 2.0, K)
        X = rng.uniform(0.0, 2.0, K)
        T_ne = float(rng.uniform(0.0, 3.0))
        t, adsf = es.maxplus_pipeline(L, X, q, b, T_ne)
        to, ao = oracle.maxplus(L, X, q, b, T_ne)
        assert t == to
        np.testing.assert_array_equal(adsf, ao)
    assert es.maxplus_pipeline([], [], 1, 1, 2.5)[0] == 2.5
    assert es.lib().estream_maxplus_pipeline(None, None, 3, 0, 1, 0.0, None) == -1.0


def _brute(profiles, T_ne, Q0, M_max, W_e, N_e):
    best = None
    for g, (L, X) in profiles.items():
        bmax = min(math.floor(M_max / (g * W_e)), -(-N_e // g))
        for b in range(Q0, bmax + 1):
            t = oracle.maxplus(L, X, Q0, b, T_ne)[0]
            if best is None or t < best[2]:
                best = (g, b, t)
    return best


def test_bank_bound_and_autoconfig(es):
    assert es.bank_bound(8, 1e9, 1e8, 12.6e6, 64) == 8
    assert es.bank_bound(8, 1e9, 0.0, 1e6, 20) == 3          # ceil(20 / 8) groups
    assert es.bank_bound(4, 1e7, 2e7, 1e6, 64) == 0          # no room
    rng = np.random.default_rng(5)
    N_e, W_e = 64, 12.6e6
    for trial in range(20):
        profiles = {}
        for g in (1, 2, 4, 8, 16):
            K = -(-N_e // g)
            # reads cost a fixed overhead plus bytes; execution grows with g
            L = 0.05 + g * W_e / 2e11 * 1e3 * rng.uniform(0.9, 1.1, K)
            X = rng.uniform(0.2, 1.0, K) * g / 8
            profiles[g] = (L, X)
        M_max = float(rng.uniform(0.5e9, 3e9))
        T_ne = float(rng.uniform(0.0, 1.0))
        want = _brute(profiles, T_ne, 1, M_max, W_e, N_e)
        G, B, T = es.autoconfig(profiles, T_ne, 1, M_max, W_e, N_e)
        assert abs(T - want[2]) < 1e-12, (G, B, T, want)
        assert oracle.maxplus(*profiles[G], 1, B, T_ne)[0] == T
    with pytest.raises(es.EStreamError):
        es.autoconfig({8: ([1.0], [1.0])}, 0.0, 2, 1e6, 1e6, 8)   # B_max(8) = 1 < Q0
