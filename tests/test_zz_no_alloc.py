"""fa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc while they run -- a host that reserves
the whole device for its own pool up front, a latency-critical loop where an
allocation could block or synchronise, a deployment that forbids allocation
after start-up.  fa_decode_noalloc keeps the split partials in a fixed array
built into the library instead.  These tests call it through the C ABI and
compare it with fa_decode_ex (the allocating entry point) on the same inputs,
twice in a row, since every call reuses the same scratch array.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import binding, build, inputs

TOL = 2e-3  # fp16 inputs (the decode tolerance used by the other decode tests)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_rejects_problems_larger_than_the_static_scratch(lib):
    # B*H*splits*(d+2)*4 bytes of partials > 4 MiB; nothing is launched.
    assert binding.fa_decode_noalloc_max_bytes() == 4 << 20
    big = binding.fa_decode_noalloc(1 << 20, 1 << 26, 1 << 27, 1 << 24, 1 << 28,
                                    4096, 64, 4096, 128, 0.1, binding.FA_F16, binding.FA_F16, 1,
                                    None)
    assert big == 8  # FA_ERR_WORKSPACE
    assert binding.fa_decode_noalloc(None, 1, 1, 1, 1, 1, 1, 64, 64, 0.1, 0, 0, 1, None) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,L,d,splits", [(8, 14, 4096, 64, 0), (3, 5, 1000, 128, 7)])
def test_noalloc_matches_allocating_decode_on_two_calls(lib, B, H, L, d, splits):
    import torch
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def tens(shape, seed):
        bits = inputs.normal_bits(shape, seed, "f16")
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16).to(dev)

    q = tens((B, H, 1, d), 41 + d)
    kc = tens((B, H, L, d), 42 + d)
    vc = tens((B, H, L, d), 43 + d)
    lens = torch.from_numpy(inputs.seq_lens(44 + d, B, L)).to(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    ref = torch.empty((B, H, 1, d), dtype=torch.float32, device=dev)
    rc = binding.fa_decode_ex(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(),
                              ref.data_ptr(), B, H, L, d, 1.0 / np.sqrt(d), binding.FA_F16,
                              binding.FA_F32, splits, None, 0, stream)
    assert rc == 0
    outs = []
    for _ in range(2):
        out = torch.full((B, H, 1, d), float("nan"), dtype=torch.float32, device=dev)
        rc = binding.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                       lens.data_ptr(), out.data_ptr(), B, H, L, d,
                                       1.0 / np.sqrt(d), binding.FA_F16, binding.FA_F32, splits,
                                       stream)
        assert rc == 0
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= TOL
