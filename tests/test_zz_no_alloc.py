"""The allocation-free route build (estream_route_build_noalloc).

It serves callers that cannot give the library device scratch memory (for
example a serving process that reserved all device memory up front and
allows no cudaMalloc on its request path). Its scratch is a static device
array shared by every call, so these tests check that two calls in a row --
with different sizes, the second one smaller -- each give exactly what the
workspace-taking estream_route_build gives, that oversized requests and
memory of the wrong kind are refused before anything runs, and that the
error word in the static array is reported and cleared by
estream_route_noalloc_error. This file is named to be collected last.
"""
import ctypes

import pytest
import torch


def _lib():
    from routed_expert_ffn_topk_gb300 import build as b
    b.build()
    from routed_expert_ffn_topk_gb300 import estream as es
    return es


def test_noalloc_rejects_null_arguments():
    es = _lib()
    L = es.lib()
    # k > E and a null offsets pointer are refused before any CUDA call
    st = L.estream_route_build_noalloc(None, 4, 8, 9, 0, None, 8, None, None, None, None, None, None)
    assert st == es.ERR_INVALID_ARG
    st = L.estream_route_build_noalloc(None, 0, 8, 2, 0, None, 8, None, None, None, None, None, None)
    assert st == es.ERR_INVALID_ARG


def _route_buffers(dev, T, k, P):
    R = T * k
    return {"topk_ids": torch.empty(R, dtype=torch.int32, device=dev),
            "alpha": torch.empty(R, dtype=torch.float32, device=dev),
            "offsets": torch.empty(P + 2, dtype=torch.int32, device=dev),
            "rec_tok": torch.empty(R, dtype=torch.int32, device=dev),
            "rec_route": torch.empty(R, dtype=torch.int32, device=dev)}


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Real device buffers of the right sizes: T=2048 tokens over P=4096 slots
    need 128 chunks x 4097 counts (about 2 MB of route scratch, beyond the
    1 MiB array) while the logits are 512 KB; the call is refused with
    ESTREAM_ERR_CAPACITY and writes nothing."""
    es = _lib()
    dev = torch.device("cuda", 0)
    T, E, k, P = 2048, 64, 1, 4096
    assert es.route_workspace_bytes(T, E, k, P) > (1 << 20)
    lg = torch.randn(T, E, generator=torch.Generator().manual_seed(5)).to(dev)
    phi = torch.arange(E, dtype=torch.int32, device=dev)
    o = _route_buffers(dev, T, k, P)
    o["offsets"].fill_(-7)
    with pytest.raises(es.EStreamError) as ex:
        es.route_build_noalloc(lg, k, False, phi, P, out=o)
    assert ex.value.status == es.ERR_CAPACITY
    torch.cuda.synchronize()
    assert bool((o["offsets"] == -7).all())


@pytest.mark.gpu
def test_noalloc_rejects_host_memory():
    """Logits in host memory are refused before any launch."""
    es = _lib()
    dev = torch.device("cuda", 0)
    T, E, k = 64, 8, 2
    lg_host = torch.randn(T, E)
    o = _route_buffers(dev, T, k, E)
    L = es.lib()
    with torch.cuda.device(dev):
        st = L.estream_route_build_noalloc(
            lg_host.data_ptr(), T, E, k, 0, None, E, o["topk_ids"].data_ptr(),
            o["alpha"].data_ptr(), o["offsets"].data_ptr(), o["rec_tok"].data_ptr(),
            o["rec_route"].data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    assert st == es.ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_route_build_twice():
    es = _lib()
    dev = torch.device("cuda", 0)
    cases = [(2048, 64, 8, True, 24), (300, 60, 4, False, 60)]   # second call smaller
    for T, E, k, renorm, P in cases:
        g = torch.Generator().manual_seed(T + E)
        lg = torch.randn(T, E, generator=g).to(dev)
        phi = None
        if P != E:
            perm = torch.randperm(E, generator=g)
            phi_h = torch.full((E,), -1, dtype=torch.int32)
            phi_h[perm[:P]] = torch.arange(P, dtype=torch.int32)
            phi = phi_h.to(dev)
        ref = es.route_build(lg, k, renorm, phi, P)
        got = es.route_build_noalloc(lg, k, renorm, phi, P)
        torch.cuda.synchronize()
        assert es.route_noalloc_error(dev) == es.OK
        R = T * k
        for name in ("topk_ids", "rec_tok", "rec_route"):
            assert torch.equal(got[name][:R], ref[name][:R]), name
        assert torch.equal(got["offsets"], ref["offsets"])
        assert torch.equal(got["alpha"][:R].view(torch.int32), ref["alpha"][:R].view(torch.int32))


@pytest.mark.gpu
def test_noalloc_reports_a_bad_slot_through_its_error_word():
    """A phi entry outside [-1, P) is filed under the trailing bucket (as the
    workspace route build does) and reported once by
    estream_route_noalloc_error; the next good call reports nothing."""
    es = _lib()
    dev = torch.device("cuda", 0)
    T, E, k, P = 256, 16, 2, 16
    lg = torch.randn(T, E, generator=torch.Generator().manual_seed(3)).to(dev)
    phi_h = torch.arange(E, dtype=torch.int32)
    phi_h[5] = P + 3                      # out of range
    phi = phi_h.to(dev)
    ref = es.route_build(lg, k, False, phi, P)
    assert es.workspace_error(ref["workspace"]) == es.ERR_DEVICE
    got = es.route_build_noalloc(lg, k, False, phi, P)
    assert es.route_noalloc_error(dev) == es.ERR_DEVICE
    assert es.route_noalloc_error(dev) == es.OK          # read and cleared
    assert torch.equal(got["offsets"], ref["offsets"])
    assert torch.equal(got["rec_route"], ref["rec_route"])
    good = es.route_build_noalloc(lg, k, False, None, E)
    assert es.route_noalloc_error(dev) == es.OK
    assert int(good["offsets"][E + 1]) == T * k
