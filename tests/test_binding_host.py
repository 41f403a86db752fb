"""The Python binding's checks of caller-supplied buffers, on the host (no GPU).

The C ABI receives bare pointers, so the binding checks every tensor it hands
over: element type, size, contiguity and device.  With host tensors, a call
whose buffers are all right gets as far as the final "CUDA device" check;
a call with a wrong buffer is refused naming that buffer.  Meta tensors stand
in for a buffer on another device.
"""
import pytest
import torch

from block_sparse_attention_nablat_gb300 import nabla as N

B, S, h, D = 1, 1024, 2, 64
s1 = S // 64
CUDA = "CUDA device"


@pytest.fixture(scope="module", autouse=True)
def lib():
    try:
        N.load()
    except RuntimeError:
        import __graft_entry__

        __graft_entry__.build()
        N.load()


def qkv(dtype=torch.bfloat16):
    return [torch.zeros(B, S, h, D, dtype=dtype) for _ in range(3)]


def csr():
    return (torch.zeros(B, h, s1, dtype=torch.int32),
            torch.zeros(B, h, s1, s1, dtype=torch.int32))


def sta():
    return torch.zeros(s1, s1, dtype=torch.uint8)


def test_valid_calls_pass_every_buffer_check():
    q, k, v = qkv()
    nb, inds = csr()
    calls = [
        lambda: N.nabla_build_mask(q, k, sta(), 0.9),
        lambda: N.nabla_build_mask(q, k, sta(), 0.9, nb, inds),
        lambda: N.nabla_build_mask_noalloc(q, k, sta(), 0.9, nb, inds),
        lambda: N.nabla_build_mask_topk(q, k, 0.1),
        lambda: N.nabla_build_mask_topk(q, k, 0.1, nb, inds),
        lambda: N.nabla_attn_fwd(q, k, v, nb, inds),
        lambda: N.nabla_attn_fwd(q, k, v, nb, inds, 0.125, torch.empty_like(q)),
        lambda: N.nabla_attn_fwd_lse(q, k, v, nb, inds),
        lambda: N.nabla_attn_bwd(q, k, v, q.clone(), q.clone(), nb, inds),
        lambda: N.nabla_attn_bwd(q, k, v, q.clone(), q.clone(), nb, inds,
                                 lse=torch.zeros(B, h, S)),
        lambda: N.nabla_fractal_flatten(torch.zeros(1, 2, 16, 16, 2, 64, dtype=torch.bfloat16), 8),
        lambda: N.nabla_fractal_unflatten(torch.zeros(1, 512, 2, 64, dtype=torch.bfloat16),
                                          2, 16, 16, 8),
        lambda: N.nabla_sta_mask(4, 2, 2, 1, 1, 1, device="cpu"),
    ]
    for call in calls:
        with pytest.raises(ValueError, match=CUDA):
            call()


def test_fp32_calls_pass_every_buffer_check():
    q, k, v = qkv(torch.float32)
    nb, inds = csr()
    with pytest.raises(ValueError, match=CUDA):
        N.nabla_attn_fwd(q, k, v, nb, inds, 0.125, torch.empty_like(q))


def test_mask_buffers_are_checked():
    q, k, _ = qkv()
    nb, inds = csr()
    with pytest.raises(ValueError, match="sta must be torch.uint8"):
        N.nabla_build_mask(q, k, sta().bool(), 0.9)
    with pytest.raises(ValueError, match="sta holds"):
        N.nabla_build_mask(q, k, sta()[:-1], 0.9)
    with pytest.raises(ValueError, match="kv_nb must be torch.int32"):
        N.nabla_build_mask(q, k, sta(), 0.9, nb.long(), inds)
    with pytest.raises(ValueError, match="kv_inds holds"):
        N.nabla_build_mask_topk(q, k, 0.1, nb, inds[..., :8].contiguous())
    with pytest.raises(ValueError, match="kv_inds must be contiguous"):
        N.nabla_build_mask_noalloc(q, k, sta(), 0.9, nb, inds.transpose(-1, -2))
    with pytest.raises(ValueError, match="workspace is on meta"):
        N.nabla_build_mask(q, k, sta(), 0.9, nb, inds,
                           torch.empty(1 << 20, dtype=torch.uint8, device="meta"))


def test_attention_buffers_are_checked():
    q, k, v = qkv()
    nb, inds = csr()
    with pytest.raises(ValueError, match="kv_nb is on meta"):
        N.nabla_attn_fwd(q, k, v, torch.empty(B, h, s1, dtype=torch.int32, device="meta"), inds)
    with pytest.raises(ValueError, match="o must be torch.bfloat16"):
        N.nabla_attn_fwd(q, k, v, nb, inds, 0.125, torch.empty(B, S, h, D))
    with pytest.raises(ValueError, match="o holds"):
        N.nabla_attn_fwd(q, k, v, nb, inds, 0.125, torch.empty(B, S // 2, h, D,
                                                               dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="v is on meta"):
        N.nabla_attn_fwd(q, k, v.to("meta"), nb, inds)
    with pytest.raises(ValueError, match="lse must be torch.float32"):
        N.nabla_attn_fwd_lse(q, k, v, nb, inds, lse=torch.zeros(B, h, S, dtype=torch.float16))
    with pytest.raises(ValueError, match="lse holds"):
        N.nabla_attn_bwd(q, k, v, q.clone(), q.clone(), nb, inds, lse=torch.zeros(B, h, S - 1))
    with pytest.raises(ValueError, match="dk must be contiguous"):
        N.nabla_attn_bwd(q, k, v, q.clone(), q.clone(), nb, inds,
                         dk=torch.zeros(B, h, S, D, dtype=torch.bfloat16).transpose(1, 2))
    with pytest.raises(ValueError, match="dout is on meta"):
        N.nabla_attn_bwd(q, k, v, q.clone(), q.to("meta"), nb, inds)


def test_fractal_and_sta_outputs_are_checked():
    x = torch.zeros(1, 2, 16, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must be torch.bfloat16"):
        N.nabla_fractal_flatten(x, 8, out=torch.empty(1, 512, 2, 64))
    with pytest.raises(ValueError, match="out holds"):
        N.nabla_fractal_flatten(x, 8, out=torch.empty(1, 256, 2, 64, dtype=torch.bfloat16))
    y = torch.zeros(1, 512, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out is on meta"):
        N.nabla_fractal_unflatten(y, 2, 16, 16, 8,
                                  out=torch.empty(1, 2, 16, 16, 2, 64, dtype=torch.bfloat16,
                                                  device="meta"))
    with pytest.raises(ValueError, match="out must be torch.uint8"):
        N.nabla_sta_mask(4, 2, 2, 1, 1, 1, out=torch.empty(16, 16, dtype=torch.int32))


def test_calls_run_with_the_tensors_device_current(monkeypatch):
    """The library launches on the current device and takes its per-device state
    from it, so the binding makes the tensors' device current for each call and
    takes the default stream from that device (not from whichever is current)."""
    seen = []

    class FakeDevice:
        def __init__(self, d):
            self.d = d

        def __enter__(self):
            seen.append(("enter", str(self.d)))

        def __exit__(self, *exc):
            seen.append(("exit", str(self.d)))

    class FakeStream:
        cuda_stream = 1234

    monkeypatch.setattr(torch.cuda, "device", FakeDevice)
    monkeypatch.setattr(torch.cuda, "current_stream",
                        lambda d=None: seen.append(("stream", str(d))) or FakeStream())
    dev = torch.device("cuda", 1)
    got = N._call(dev, lambda *a: seen.append(("call", a)) or 0, N._stream(None, dev))
    assert got == 0
    assert seen == [("stream", "cuda:1"), ("enter", "cuda:1"), ("call", (1234,)),
                    ("exit", "cuda:1")]
