"""K1 (router top-k + route map) against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(logits_np, k, renorm, phi=None, P=None):
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = torch.device("cuda", 0)
    lg = torch.from_numpy(np.ascontiguousarray(logits_np, dtype=np.float32)).to(dev)
    ph = None if phi is None else torch.as_tensor(phi, dtype=torch.int32).to(dev)
    out = es.route_build(lg, k, renorm, ph, P)
    assert es.workspace_error(out["workspace"]) == es.OK
    T, E = logits_np.shape
    R = T * k
    return {n: out[n].cpu().numpy()[:R] if n != "offsets" else out[n].cpu().numpy()
            for n in ("topk_ids", "alpha", "offsets", "rec_tok", "rec_route")}


def _check(logits_np, k, renorm, phi=None, P=None):
    T, E = logits_np.shape
    P = E if P is None else P
    got = _run(logits_np, k, renorm, phi, P)
    ids, alpha = oracle.route_topk(logits_np, k, renorm)
    offs, rt, rr = oracle.route_csr(ids, E, P, phi)
    np.testing.assert_array_equal(got["topk_ids"], ids.ravel())
    np.testing.assert_array_equal(got["alpha"].view(np.uint32), alpha.ravel().view(np.uint32))
    np.testing.assert_array_equal(got["offsets"], offs)
    np.testing.assert_array_equal(got["rec_tok"], rt)
    np.testing.assert_array_equal(got["rec_route"], rr)


@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c4", "c5"])
def test_route_parity_configs(key):
    cfg = W.CONFIGS[key]
    wl = W.make_workload(cfg, weights=False)
    for lg in wl.logits:
        _check(lg.numpy(), cfg.k, cfg.renorm)


@pytest.mark.parametrize("T,E,k,renorm", [(1, 1, 1, 0), (1, 5, 5, 1), (129, 8, 2, 1),
                                          (1000, 64, 8, 0), (333, 60, 6, 1), (77, 256, 16, 1),
                                          (9, 1024, 32, 0), (2049, 16, 3, 0)])
def test_route_parity_shapes(T, E, k, renorm):
    rng = np.random.default_rng(T * 1000 + E)
    _check(rng.standard_normal((T, E)).astype(np.float32) * 3, k, renorm)


def test_route_adversarial_logits():
    rng = np.random.default_rng(5)
    T, E, k = 300, 32, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0:40] = 0.5                                  # all-equal rows
    lg[40:80, 7] = 60.0                             # one expert takes everything
    lg[80:120] = np.round(lg[80:120])               # many ties
    lg[120:160] *= 80.0                             # exponent underflow for most experts
    lg[160:200, :] = lg[160:161, :]                 # identical rows
    lg[200:240] = 0.0
    lg[200:240, ::3] = -0.0                         # signed zeros compare equal: id order decides
    lg[240:260, ::2] = -0.0
    lg[240:260, 1::4] = 1e-30                       # tiny positives above both zeros
    for renorm in (0, 1):
        _check(lg, k, renorm)


def test_route_partial_placement_and_bottom_bucket():
    rng = np.random.default_rng(6)
    T, E, k, P = 500, 64, 8, 16
    lg = rng.standard_normal((T, E)).astype(np.float32)
    phi = -np.ones(E, dtype=np.int32)
    chosen = rng.choice(E, size=P, replace=False)
    phi[chosen] = rng.permutation(P)
    _check(lg, k, 0, phi, P)
    # Eq. 4 placement of grouped experts as phi
    perm = rng.permutation(E).astype(np.int32)
    bank = -np.ones(E // 8, dtype=np.int32)
    bank[[1, 5]] = [1, 0]
    phi4 = oracle.grouped_placement(perm, E, 8, bank)
    _check(lg, k, 1, phi4, 16)
    # nothing resident: every route in the trailing bucket
    _check(lg, k, 0, -np.ones(E, dtype=np.int32), 0)


def test_route_bad_phi_reported():
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = torch.device("cuda", 0)
    lg = torch.randn(64, 8, device=dev)
    phi = torch.tensor([0, 1, 2, 3, 9, 5, 6, 7], dtype=torch.int32, device=dev)  # 9 >= P
    out = es.route_build(lg, 2, False, phi, 8)
    assert es.workspace_error(out["workspace"]) == es.ERR_DEVICE
    assert es.workspace_error(out["workspace"]) == es.OK   # cleared
