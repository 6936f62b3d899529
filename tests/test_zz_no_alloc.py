"""The entry point for callers that cannot allocate device memory.

dory_q8_quantize_noalloc quantises K/V rows into q8_2f codes, scales and fields with its
working memory in a static device array instead of cudaMalloc. Its output must match,
bit for bit, what the regular path (dory_write_kv_rows into an empty slot, read back
with dory_read_kv_q8) stores for the same rows. The calls come several in a row on the
same static array (a later call must not see an earlier one's state), over the limits the
entry point accepts: 16 KV heads of 128 channels (the whole array), one head of 32
channels (a V group of one warp), and 2 heads of 64; n = 1 and 64 (nothing freezes, the
fields stay zero), 65 (the freeze comes with the last row), 66 and 300. This file sorts
last so that a failure here comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

ROWS = (1, 64, 65, 66, 300)


def _noalloc(lib, k, v, torch):
    n, nk, hd = k.shape
    dev = "cuda:0"
    kd = torch.from_numpy(k).to(dev)
    vd = torch.from_numpy(v).to(dev)
    kq = torch.empty((nk, n, hd), dtype=torch.int8, device=dev)
    ks = torch.empty((nk, n, hd // 32), dtype=torch.float32, device=dev)
    vq = torch.empty((nk, n, hd), dtype=torch.int8, device=dev)
    vs = torch.empty((nk, n), dtype=torch.float32, device=dev)
    kcol = torch.full((nk, hd), 7.0, dtype=torch.float32, device=dev)  # must come back zero or frozen
    vcol = torch.full((nk, hd), 7.0, dtype=torch.float32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.dory_q8_quantize_noalloc(p(kd), p(vd), n, nk, hd, p(kq), p(ks), p(vq), p(vs), p(kcol), p(vcol), None)
    assert rc == 0, lib.dory_last_error()
    torch.cuda.synchronize()
    return {name: t.cpu().numpy() for name, t in
            dict(kq=kq, ks=ks, vq=vq, vs=vs, kcol=kcol, vcol=vcol).items()}


@pytest.mark.parametrize("nk,hd", [(16, 128), (1, 32), (2, 64)])
def test_the_no_alloc_quantiser_matches_the_regular_append(nk, hd):
    torch = pytest.importorskip("torch")
    from looped_normalized_gpt_gb300 import Dory, build, load_library

    build()
    lib = load_library()
    nh = 16 if nk == 16 else 8
    cfg = synth.small(kv_quant="q8_2f", nh=nh, nk=nk, hd=hd, max_seqs=2)
    g = Dory(cfg, synth.weights(cfg, 3001))
    try:
        for call, n in enumerate(ROWS):
            scale = (3.0, 0.5, 1.0, 2.0, 0.25)[call]
            k = synth.kv_rows(3001, 10 + call, n, nk, hd) * np.float32(scale)
            v = synth.kv_rows(3001, 20 + call, n, nk, hd) * np.linspace(0.2, 5, hd).astype(np.float32)
            got = _noalloc(lib, k, v, torch)
            seq = call % 2
            g.reset(seq)
            g.write_kv_rows(seq, 0, 0, 0, k, v)
            want = g.read_kv_q8(seq, 0, 0)
            frozen = n > 64
            assert want["frozen"].tolist() == [int(frozen)] * nk
            assert np.array_equal(got["kq"], want["kq"][:, :n]), (n, "kq")
            assert np.array_equal(got["vq"], want["vq"][:, :n]), (n, "vq")
            assert np.array_equal(got["ks"].view(np.uint32), want["ks"][:, :n].view(np.uint32)), (n, "ks")
            assert np.array_equal(got["vs"].view(np.uint32), want["vs"][:, :n].view(np.uint32)), (n, "vs")
            assert np.array_equal(got["kcol"].view(np.uint32), want["kcol"].view(np.uint32)), (n, "kcol")
            assert np.array_equal(got["vcol"].view(np.uint32), want["vcol"].view(np.uint32)), (n, "vcol")
            if not frozen:
                assert not got["kcol"].any() and not got["vcol"].any()
    finally:
        g.close()


def test_sizes_beyond_the_static_array_are_refused():
    """More KV heads than the array holds, or an unsupported head width, is DORY_EINVAL with
    a message, before anything is queued."""
    pytest.importorskip("torch")
    from looped_normalized_gpt_gb300 import build, load_library

    build()
    lib = load_library()
    dummy = ctypes.c_void_p(16)  # never dereferenced: the sizes are checked first
    for n, nk, hd in [(10, 17, 128), (10, 2, 256), (10, 2, 48), (0, 2, 64)]:
        rc = lib.dory_q8_quantize_noalloc(dummy, dummy, n, nk, hd, *[dummy] * 6, None)
        assert rc == -1, (n, nk, hd)
        assert lib.dory_last_error()
