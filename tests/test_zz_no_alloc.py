"""The entry point for callers that cannot allocate device memory.

dory_q8_quantize_noalloc quantises K/V rows into q8_2f codes, scales and fields with its
working memory in a static device array instead of cudaMalloc. Its output must match,
bit for bit, what the regular path (dory_write_kv_rows into an empty slot, read back
with dory_read_kv_q8) stores for the same rows, on two calls in a row (the second call
must not see the first one's state). This file sorts last so that a failure here comes
after every other test has run.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _noalloc(lib, k, v, torch):
    n, nk, hd = k.shape
    dev = "cuda:0"
    kd = torch.from_numpy(k).to(dev)
    vd = torch.from_numpy(v).to(dev)
    kq = torch.empty((nk, n, hd), dtype=torch.int8, device=dev)
    ks = torch.empty((nk, n, hd // 32), dtype=torch.float32, device=dev)
    vq = torch.empty((nk, n, hd), dtype=torch.int8, device=dev)
    vs = torch.empty((nk, n), dtype=torch.float32, device=dev)
    kcol = torch.empty((nk, hd), dtype=torch.float32, device=dev)
    vcol = torch.empty((nk, hd), dtype=torch.float32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.dory_q8_quantize_noalloc(p(kd), p(vd), n, nk, hd, p(kq), p(ks), p(vq), p(vs), p(kcol), p(vcol), None)
    assert rc == 0, lib.dory_last_error()
    torch.cuda.synchronize()
    return {name: t.cpu().numpy() for name, t in
            dict(kq=kq, ks=ks, vq=vq, vs=vs, kcol=kcol, vcol=vcol).items()}


def _regular(cfg, w, k, v, seq):
    from looped_normalized_gpt_gb300 import Dory

    g = Dory(cfg, w)
    try:
        g.write_kv_rows(seq, 0, 0, 0, k, v)
        return g.read_kv_q8(seq, 0, 0)
    finally:
        g.close()


def test_the_no_alloc_quantiser_matches_the_regular_append_twice():
    torch = pytest.importorskip("torch")
    from looped_normalized_gpt_gb300 import build, load_library

    build()
    lib = load_library()
    cfg = synth.small(kv_quant="q8_2f", max_seqs=2)
    w = synth.weights(cfg, 3001)
    for call, (n, scale) in enumerate([(300, 3.0), (100, 0.5)]):
        k = synth.kv_rows(3001, 10 + call, n, cfg.nk, cfg.hd) * np.float32(scale)
        v = synth.kv_rows(3001, 20 + call, n, cfg.nk, cfg.hd) * np.linspace(0.2, 5, cfg.hd).astype(np.float32)
        got = _noalloc(lib, k, v, torch)
        want = _regular(cfg, w, k, v, seq=call % 2)
        assert want["frozen"].tolist() == [1] * cfg.nk
        assert np.array_equal(got["kq"], want["kq"][:, :n])
        assert np.array_equal(got["vq"], want["vq"][:, :n])
        assert np.array_equal(got["ks"].view(np.uint32), want["ks"][:, :n].view(np.uint32))
        assert np.array_equal(got["vs"].view(np.uint32), want["vs"][:, :n].view(np.uint32))
        assert np.array_equal(got["kcol"].view(np.uint32), want["kcol"].view(np.uint32))
        assert np.array_equal(got["vcol"].view(np.uint32), want["vcol"].view(np.uint32))
