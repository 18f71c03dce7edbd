"""GPU parity of prefill on host buffers (fa_prefill_host through the binding):
the copies in, the kernels on chunks of key/value heads and the copies out
against the fp64 oracle, and bit for bit against the device-buffer call when
both run the unit schedule (every unit whole in one CTA, so cutting the heads
into chunks cannot change a bit).
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import torch
    from attention_forward_prefill_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    assert binding.fa_device_status(True) == 0
    yield binding
    assert binding.fa_device_status(False) == 0, "a kernel watchdog fired"


def host_tensor(bits, dtype, pinned):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(G.torch_dtype(dtype))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("shape,causal,pinned,out_dtype", [
    ((2, 4, 2, 300, 700, 64), True, True, "f32"),       # one chunk (under 8 MB), chunk prompt
    ((1, 6, 6, 8192, 8192, 128), False, True, "f32"),   # chunks of 1, 2, 2 and 1 heads
    ((1, 16, 4, 4096, 4096, 64), True, True, "bf16"),   # grouped heads, two chunks of 2 KV heads
    ((2, 6, 2, 1500, 1500, 64), True, False, "f16"),    # pageable memory, grouped heads
])
def test_host_buffers_match_the_oracle(fa, oracle_mod, shape, causal, pinned, out_dtype):
    B, Hq, Hkv, Nq, Nk, d = shape
    dtype = "bf16" if d == 128 else "f16"
    q = inputs.normal_bits((B, Hq, Nq, d), 1500 + Nq, dtype)
    k = inputs.normal_bits((B, Hkv, Nk, d), 1501 + Nq, dtype)
    v = inputs.normal_bits((B, Hkv, Nk, d), 1502 + Nq, dtype)
    scale = 1.0 / np.sqrt(d)
    out = fa.prefill(*(host_tensor(x, dtype, pinned) for x in (q, k, v)), causal=causal,
                     scale=scale, out_dtype=G.torch_dtype(out_dtype))
    assert not out.is_cuda and out.is_pinned() == pinned
    got = out.float().numpy().astype(np.float64)
    rows = G.sample_rows(Nq, 19) if Nq > 1024 else None
    qf, kf, vf = (oracle_mod.bits_to_f64(x, dtype) for x in (q, k, v))
    want = oracle_mod.attention(qf, kf, vf, causal, scale, rows=rows, threads=G.THREADS)
    if rows is not None:
        got = got[:, :, rows]
    G.assert_close(got, want, dtype, out_dtype, f"host prefill {shape} causal={causal}")


def test_host_buffers_equal_the_device_call_bit_for_bit(fa):
    # four key/value heads of 8192 keys: chunks of 1, 2 and 1 heads
    import torch
    B, Hq, Hkv, N, d = 2, 8, 2, 8192, 128
    q, k, v = (inputs.normal_bits((B, h, N, d), 1600 + i, "bf16") for i, h in enumerate((Hq, Hkv, Hkv)))
    hq, hk, hv = (host_tensor(x, "bf16", True) for x in (q, k, v))
    for causal in (False, True):
        flags = fa.FA_FLAG_SCHEDULE_UNITS
        host_out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, pin_memory=True)
        got = fa.prefill(hq, hk, hv, causal=causal, scale=0.088, flags=flags, out=host_out)
        assert got.data_ptr() == host_out.data_ptr()
        dev = fa.prefill(hq.cuda(), hk.cuda(), hv.cuda(), causal=causal, scale=0.088, flags=flags)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), dev.cpu().view(torch.int16))


def test_host_buffers_repeat_on_a_side_stream(fa):
    # the call is ordered on the current stream, whichever it is
    import torch
    q, k, v = (host_tensor(inputs.normal_bits((1, 4, 1024, 64), 1700 + i, "f16"), "f16", True)
               for i in range(3))
    ref = fa.prefill(q, k, v, causal=True, scale=0.125)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = [fa.prefill(q, k, v, causal=True, scale=0.125) for _ in range(3)]
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def test_host_buffers_asynchronous_on_several_streams(fa):
    # sync=False: the calls return at once; after a device synchronisation every
    # output equals the synchronous call's
    import torch
    shapes = [(1, 4, 1024, 64), (1, 8, 2048, 64), (2, 4, 512, 64)]
    ins = [[host_tensor(inputs.normal_bits(sh, 1800 + 3 * n + i, "f16"), "f16", True) for i in range(3)]
           for n, sh in enumerate(shapes)]
    refs = [fa.prefill(*x, causal=True, scale=0.125) for x in ins]
    outs = [torch.empty(sh, dtype=torch.float16, pin_memory=True) for sh in shapes]
    streams = [torch.cuda.Stream() for _ in shapes]
    for _ in range(2):
        for x, o, s in zip(ins, outs, streams):
            with torch.cuda.stream(s):
                fa.prefill(*x, causal=True, scale=0.125, out=o, sync=False)
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
