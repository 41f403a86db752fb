"""Programmatic dependent launch on and off give the same results (GPU).

NABLA_DISABLE_PDL is read once per process, so the plain-launch run happens in a
child process; both runs compute one small step (mask build, forward with
log-sum-exp, backward) on the same seeded inputs and must agree bit for bit.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from block_sparse_attention_nablat_gb300 import nabla, workloads as W
w = W.custom("pdl", 1, 2, 128, 64 * 24, (6, 2, 2), sigma=0.75, rho=0.8)
data = W.generate(w, 3)
q, k, v = (nabla.from_storage(data[n], "cuda:0") for n in "qkv")
g = nabla.from_storage(W.generate_dout(w, 3), "cuda:0")
sta = nabla.nabla_sta_mask(*w.grid, 1, 1, 1, device="cuda:0")
nb, inds = nabla.nabla_build_mask(q, k, sta, 0.8)
o, lse = nabla.nabla_attn_fwd_lse(q, k, v, nb, inds, w.scale)
dq, dk, dv = nabla.nabla_attn_bwd(q, k, v, o, g, nb, inds, w.scale, lse=lse)
assert nabla.nabla_get_last_device_status() == 0
n = nb.cpu().numpy()
out = {"nb": n, "o": o.float().cpu().numpy(), "lse": lse.cpu().numpy(),
       "dq": dq.float().cpu().numpy(), "dk": dk.float().cpu().numpy(),
       "dv": dv.float().cpu().numpy()}
ii = inds.cpu().numpy()
out["inds"] = np.where(np.arange(ii.shape[-1]) < n[..., None], ii, -1)
np.savez(sys.argv[2], **out)
"""


def _run(tmp_path, disable):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    from block_sparse_attention_nablat_gb300 import nabla

    try:
        nabla.load()
    except RuntimeError:
        __graft_entry__.build()
    env = dict(os.environ, NABLA_DISABLE_PDL="1" if disable else "0")
    path = str(tmp_path / f"out_{int(disable)}.npz")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return dict(np.load(path))


def test_plain_and_chained_launches_agree(tmp_path):
    a = _run(tmp_path, False)
    b = _run(tmp_path, True)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
