"""The C ABI on the host, without a GPU: the library loads, exports every entry
point include/nabla.h declares, sizes the workspace, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "block_sparse_attention_nablat_gb300", "libnabla.so")
HEADER = os.path.join(ROOT, "include", "nabla.h")

INVALID = 1


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__

        __graft_entry__.build()
    from block_sparse_attention_nablat_gb300 import nabla

    return nabla.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nabla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["nabla_build_mask", "nabla_build_mask_topk", "nabla_attn_fwd", "nabla_sta_mask",
              "nabla_build_mask_workspace_bytes", "nabla_get_last_device_status",
              "nabla_status_string", "nabla_abi_version"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.nabla_abi_version() == 1
    for code, name in enumerate(["NABLA_OK", "NABLA_ERR_INVALID_ARG", "NABLA_ERR_UNSUPPORTED",
                                 "NABLA_ERR_CUDA", "NABLA_ERR_TIMEOUT", "NABLA_ERR_BAD_INDEX"]):
        assert lib.nabla_status_string(code).decode() == name
    assert lib.nabla_status_string(99).decode() == "NABLA_ERR_UNKNOWN"


def _ws(B, S, h, D):
    s1 = S // 64

    def up(x):
        return (x + 255) // 256 * 256

    means = up(B * h * s1 * D * 4)
    return up(4 * means + B * h * s1 * s1 * 4)


@pytest.mark.parametrize("shape", [(1, 1024, 2, 64), (1, 98304, 24, 128), (2, 64 * 37, 3, 128)])
def test_workspace_bytes(lib, shape):
    assert lib.nabla_build_mask_workspace_bytes(*shape) == _ws(*shape)


@pytest.mark.parametrize("shape", [(1, 1000, 2, 64), (1, 1024, 2, 96), (0, 1024, 2, 64),
                                   (1, 1024, 0, 64), (1, 64 * 2049, 1, 64), (1, 0, 2, 64)])
def test_workspace_bytes_rejects_bad_shapes(lib, shape):
    assert lib.nabla_build_mask_workspace_bytes(*shape) == 0


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: arguments fail validation first


def _mask(lib, **kw):
    a = dict(q=FAKE, k=FAKE, dt=1, B=1, S=1024, h=2, D=64, sta=FAKE, thr=0.9, nb=FAKE,
             inds=FAKE, ws=FAKE, wsb=1 << 30, st=None)
    a.update(kw)
    return lib.nabla_build_mask(a["q"], a["k"], a["dt"], a["B"], a["S"], a["h"], a["D"],
                                a["sta"], a["thr"], a["nb"], a["inds"], a["ws"], a["wsb"],
                                a["st"])


@pytest.mark.parametrize("kw", [dict(S=1000), dict(D=96), dict(B=0), dict(h=0),
                                dict(S=64 * 2049), dict(thr=0.0), dict(thr=1.5),
                                dict(thr=float("nan")), dict(thr=-0.1), dict(q=None),
                                dict(k=None), dict(sta=None), dict(nb=None), dict(inds=None),
                                dict(ws=None), dict(q=FAKE + 8), dict(ws=FAKE + 16),
                                dict(nb=FAKE + 2), dict(wsb=100), dict(dt=7)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_build_mask_rejects(lib, kw):
    assert _mask(lib, **kw) == INVALID


def _topk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, dt=1, B=1, S=1024, h=2, D=64, ratio=0.25, nb=FAKE, inds=FAKE,
             ws=FAKE, wsb=1 << 30, st=None)
    a.update(kw)
    return lib.nabla_build_mask_topk(a["q"], a["k"], a["dt"], a["B"], a["S"], a["h"], a["D"],
                                     a["ratio"], a["nb"], a["inds"], a["ws"], a["wsb"], a["st"])


@pytest.mark.parametrize("kw", [dict(S=1000), dict(D=96), dict(B=0), dict(h=0),
                                dict(ratio=-0.1), dict(ratio=float("nan")),
                                dict(ratio=float("inf")), dict(q=None), dict(k=None),
                                dict(nb=None), dict(inds=None), dict(ws=None), dict(k=FAKE + 8),
                                dict(ws=FAKE + 16), dict(inds=FAKE + 2), dict(wsb=100),
                                dict(dt=7)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_build_mask_topk_rejects(lib, kw):
    assert _topk(lib, **kw) == INVALID


def _attn(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=1, B=1, S=1024, h=2, D=64, nb=FAKE, inds=FAKE,
             scale=0.125, o=FAKE, st=None)
    a.update(kw)
    return lib.nabla_attn_fwd(a["q"], a["k"], a["v"], a["dt"], a["B"], a["S"], a["h"], a["D"],
                              a["nb"], a["inds"], a["scale"], a["o"], a["st"])


@pytest.mark.parametrize("kw", [dict(S=1000), dict(D=32), dict(B=0), dict(v=None), dict(o=None),
                                dict(nb=None), dict(inds=None), dict(o=FAKE + 4),
                                dict(scale=float("inf")), dict(scale=float("nan")), dict(dt=2)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_attn_rejects(lib, kw):
    assert _attn(lib, **kw) == INVALID


def _bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, g=FAKE, dt=1, B=1, S=1024, h=2, D=64,
             nb=FAKE, inds=FAKE, scale=0.125, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE, wsb=1 << 30,
             st=None)
    a.update(kw)
    return lib.nabla_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["g"], a["dt"], a["B"],
                              a["S"], a["h"], a["D"], a["nb"], a["inds"], a["scale"], a["dq"],
                              a["dk"], a["dv"], a["ws"], a["wsb"], a["st"])


def test_attn_fwd_lse_rejects(lib):
    args = [FAKE, FAKE, FAKE, 1, 1, 1024, 2, 64, FAKE, FAKE, 0.125, FAKE]
    assert lib.nabla_attn_fwd_lse(*args, None, None) == INVALID       # lse required
    assert lib.nabla_attn_fwd_lse(*args, FAKE + 2, None) == INVALID   # lse misaligned
    bad = list(args)
    bad[5] = 1000
    assert lib.nabla_attn_fwd_lse(*bad, FAKE, None) == INVALID


@pytest.mark.parametrize("kw", [dict(S=1000), dict(D=32), dict(B=0), dict(o=None), dict(g=None),
                                dict(dq=None), dict(dk=FAKE + 4), dict(dv=None), dict(ws=None),
                                dict(ws=FAKE + 64), dict(wsb=1000), dict(nb=FAKE + 2),
                                dict(scale=float("nan")), dict(dt=3), dict(lse=FAKE + 2), dict(lse=FAKE + 8)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_attn_bwd_rejects(lib, kw):
    assert _bwd(lib, **kw) == INVALID


@pytest.mark.parametrize("shape", [(1, 1024, 2, 64), (1, 98304, 24, 128), (2, 64 * 37, 3, 128)])
def test_attn_bwd_workspace_bytes(lib, shape):
    B, S, h, D = shape
    s1 = S // 64

    def up(x):
        return (x + 255) // 256 * 256

    want = 2 * up(B * h * S * 4) + up(B * h * s1 * 4) + up(B * h * s1 * s1 * 4) + \
        up(B * h * s1 * ((s1 + 31) // 32) * 4) + up(B * S * h * D * 2)
    assert lib.nabla_attn_bwd_workspace_bytes(*shape) == want
    assert lib.nabla_attn_bwd_workspace_bytes(1, 1000, 2, 64) == 0


@pytest.mark.parametrize("args", [(0, 2, 2, 1, 1, 1), (4, 2, 2, -1, 1, 1), (64, 8, 8, 1, 1, 1)])
def test_sta_rejects(lib, args):
    assert lib.nabla_sta_mask(*args, FAKE, None) == INVALID
    assert lib.nabla_sta_mask(4, 2, 2, 1, 1, 1, None, None) == INVALID


def _fractal(lib, flatten, **kw):
    a = dict(src=FAKE, dt=1, B=1, T=2, H=16, W=16, h=2, D=64, P=8, dst=FAKE + (1 << 32), st=None)
    a.update(kw)
    fn = lib.nabla_fractal_flatten if flatten else lib.nabla_fractal_unflatten
    return fn(a["src"], a["dt"], a["B"], a["T"], a["H"], a["W"], a["h"], a["D"], a["P"],
              a["dst"], a["st"])


@pytest.mark.parametrize("flatten", [True, False], ids=["flatten", "unflatten"])
@pytest.mark.parametrize("kw", [dict(dt=7), dict(B=0), dict(T=0), dict(H=0), dict(P=0),
                                dict(H=12), dict(W=20), dict(h=1, D=3), dict(src=None),
                                dict(dst=None), dict(src=FAKE + 8), dict(dst=FAKE + (1 << 32) + 4),
                                dict(dst=FAKE + 16)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_fractal_rejects(lib, flatten, kw):
    """Ragged patches, rows that are not whole 16-byte chunks, NULL, unaligned and
    overlapping buffers are refused on the host, before any launch."""
    assert _fractal(lib, flatten, **kw) == INVALID


def test_product_path_has_no_oracle_dependency():
    """The package and its native sources never import or link the oracle."""
    pkg = os.path.join(ROOT, "block_sparse_attention_nablat_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|nabla_oracle|"
                                     r"oracle[/\\])", text), f
