"""fa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc while they run -- a host that reserves
the whole device for its own pool up front, a latency-critical loop where an
allocation could block or synchronise, a deployment that forbids allocation
after start-up.  fa_decode_noalloc keeps the split partials in a fixed array
built into the library instead.  These tests call it through the C ABI and
compare it with fa_decode_ex (the allocating entry point) at the same split
count: the two run the same kernels on the same partial layout, so their
outputs must be the same bits.  Every call reuses the one scratch array, so
the test makes two calls in a row with a call of another shape between
them, checks both against the fp64 oracle, and checks that the library's
scratch pool saw no allocation meanwhile.

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
    assert big == binding.FA_ERR_WORKSPACE
    assert binding.fa_decode_noalloc(None, 1, 1, 1, 1, 1, 1, 64, 64, 0.1, 0, 0, 1, None) == \
        binding.FA_ERR_NULL


class Problem:
    """Seeded decode inputs on the device, the split count, and the oracle."""

    def __init__(self, B, H, L, d, splits, seed):
        import torch
        self.B, self.H, self.L, self.d = B, H, L, d
        self.splits = splits or binding.fa_decode_choose_splits(B, H, L, -1)
        self.bits = [inputs.normal_bits(s, seed + i, "f16")
                     for i, s in enumerate(((B, H, 1, d), (B, H, L, d), (B, H, L, d)))]
        self.lens = inputs.seq_lens(seed + 3, B, L)
        self.q, self.kc, self.vc = (
            torch.from_numpy(b.view(np.int16).copy()).view(torch.float16).cuda() for b in self.bits)
        self.ld = torch.from_numpy(self.lens).cuda()
        self.scale = 1.0 / np.sqrt(d)

    def args(self, out):
        return (self.q.data_ptr(), self.kc.data_ptr(), self.vc.data_ptr(), self.ld.data_ptr(),
                out.data_ptr(), self.B, self.H, self.L, self.d, self.scale, binding.FA_F16,
                binding.FA_F32)

    def new_out(self):
        import torch
        return torch.full((self.B, self.H, 1, self.d), float("nan"), dtype=torch.float32,
                          device="cuda")

    def oracle(self, oracle_mod):
        f = [oracle_mod.bits_to_f64(b, "f16") for b in self.bits]
        return oracle_mod.decode(*f, self.lens, self.scale)


@pytest.mark.gpu
def test_noalloc_matches_allocating_decode_on_two_calls(lib, oracle_mod):
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    a = Problem(8, 14, 4096, 64, 0, 41)     # the library's own split choice
    b = Problem(3, 5, 1000, 128, 7, 51)     # another shape and split count in between
    assert binding.fa_decode_workspace_bytes(a.B, a.H, a.L, a.d, a.splits) <= \
        binding.fa_decode_noalloc_max_bytes()

    # the allocating entry point, at the same split counts
    refs = []
    for p in (a, b):
        out = p.new_out()
        assert binding.fa_decode_ex(*p.args(out), p.splits, None, 0, stream) == binding.FA_OK
        refs.append(out)
    torch.cuda.synchronize()
    rc, before = binding.fa_pool_stats(reset_high=True)
    assert rc == binding.FA_OK

    outs = []
    for p in (a, b, a):
        out = p.new_out()
        assert binding.fa_decode_noalloc(*p.args(out), p.splits, stream) == binding.FA_OK
        outs.append(out)
    torch.cuda.synchronize()
    rc, after = binding.fa_pool_stats()
    assert rc == binding.FA_OK
    # nothing was taken from the library's pool while the three calls ran
    assert after[3] <= before[2] and after[2] == before[2]

    want_a, want_b = a.oracle(oracle_mod), b.oracle(oracle_mod)
    for out, ref, want in ((outs[0], refs[0], want_a), (outs[1], refs[1], want_b),
                           (outs[2], refs[0], want_a)):
        assert torch.equal(out, ref)           # same kernels, same split: same bits
        got = out.cpu().numpy().astype(np.float64)
        assert np.abs(got - want).max() <= TOL
