"""nabla_build_mask_noalloc, the mask builder for callers that cannot allocate
device memory (an engine that owns all device memory after start-up, a loop that
cannot afford the synchronisation an allocation may imply, a plug-in without a
memory budget of its own).  It keeps its scratch in a fixed device array of the
library instead of a caller workspace, and must give exactly what
nabla_build_mask gives.  This file is collected last on purpose: the GPU test
here also has to pass after every other test has run in the same process."""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_nablat_gb300 import workloads as W

LIMIT = 64 << 20  # NABLA_NOALLOC_SCRATCH_BYTES
OK, INVALID, UNSUPPORTED = 0, 1, 2


def _lib():
    from block_sparse_attention_nablat_gb300 import nabla

    try:
        return nabla, nabla.load()
    except RuntimeError:
        import __graft_entry__

        __graft_entry__.build()
        return nabla, nabla.load()


def _call(lib, q, k, dt, shape, sta, thr, nb, inds, stream=None):
    B, S, h, D = shape
    return lib.nabla_build_mask_noalloc(q, k, dt, B, S, h, D, sta, thr, nb, inds, stream)


def test_noalloc_rejects_on_the_host():
    """Shapes past the fixed scratch and bad arguments are refused before any
    device work (so this runs without a GPU)."""
    _, lib = _lib()
    fake = 1 << 20
    big = (1, 98304, 24, 128)  # 720p-like: four 18.9 MB mean arrays + a 226 MB map
    need = lib.nabla_build_mask_workspace_bytes(*big)
    assert need > LIMIT and abs(need - 301.7e6) < 1e6, need
    assert _call(lib, fake, fake, 1, big, fake, 0.9, fake, fake) == UNSUPPORTED
    assert _call(lib, fake, fake, 1, (1, 1000, 2, 64), fake, 0.9, fake, fake) == INVALID
    assert _call(lib, fake, fake, 1, (1, 1024, 2, 64), fake, 0.0, fake, fake) == INVALID
    assert _call(lib, None, fake, 1, (1, 1024, 2, 64), fake, 0.9, fake, fake) == INVALID
    assert _call(lib, fake, fake, 5, (1, 1024, 2, 64), fake, 0.9, fake, fake) == INVALID


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls():
    """Two calls in a row with different shapes and inputs, each compared with
    nabla_build_mask on the same inputs: the kept counts and the kept index
    lists must be identical (same kernels, so bit-exact)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nabla, lib = _lib()
    dev = torch.device("cuda:0")
    cases = [(W.WORKLOADS["small_bf16"], 0, 0.9),
             (W.custom("noalloc2", 2, 3, 64, 64 * 40, (5, 2, 4), sigma=0.75, rho=0.8), 7, 0.7)]
    for w, seed, thr in cases:
        d = W.generate(w, seed)
        q, k = nabla.from_storage(d["q"], dev), nabla.from_storage(d["k"], dev)
        sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=dev)
        ref_nb, ref_inds = nabla.nabla_build_mask(q, k, sta, thr)
        nb = torch.full((w.B, w.h, w.s1), -1, dtype=torch.int32, device=dev)
        inds = torch.full((w.B, w.h, w.s1, w.s1), -1, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated(dev)
        free = torch.cuda.mem_get_info(dev)[0]
        st = _call(lib, q.data_ptr(), k.data_ptr(), 1 if w.dtype == "bf16" else 0,
                   (w.B, w.S, w.h, w.D), sta.data_ptr(), thr, nb.data_ptr(), inds.data_ptr(),
                   torch.cuda.current_stream().cuda_stream)
        assert st == OK
        assert nabla.nabla_get_last_device_status() == 0
        # nothing was allocated: torch's pool is untouched, and from the second call on
        # (the first may be what loads the library's static array, with lazy module
        # loading) the device's free memory is what it was before the call
        assert torch.cuda.memory_allocated(dev) == allocated
        if w is not cases[0][0]:
            assert torch.cuda.mem_get_info(dev)[0] == free
        a_nb, b_nb = ref_nb.cpu().numpy(), nb.cpu().numpy()
        assert np.array_equal(a_nb, b_nb)
        a, b = ref_inds.cpu().numpy(), inds.cpu().numpy()
        keep = np.arange(w.s1)[None, None, None, :] < a_nb[..., None]
        assert np.array_equal(np.where(keep, a, -1), np.where(keep, b, -1))
