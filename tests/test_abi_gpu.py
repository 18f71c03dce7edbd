"""The C entry points themselves on the GPU, with raw device pointers.

The plain calls fa_prefill / fa_decode (fp16 in, fp16 out, the pages' usage
in the flash-attention-cuda README, "Installation") and fa_prefill_ex /
fa_decode_ex are called through ctypes exactly as a C caller would, and
compared element by element with the fp64 oracle on the target's workloads.
The device status word is exercised both ways it can be set: by clamped
lengths (FA_ERR_SEQ_LEN) and by a bounded wait that runs out
(FA_ERR_WATCHDOG, through the library's self-test kernel, which has nothing
else in flight).  Also the read-bandwidth probe's checksum and the scratch
pool counters.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

CFG_TINY, CFG_GPT2, CFG_LONG, CFG_DECODE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def fa():
    import torch
    from attention_forward_prefill_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3), "libfa_gb300 targets sm_103a"
    build.build()
    binding.load()
    assert binding.fa_device_status(True) == 0
    yield binding
    assert binding.fa_device_status(False) == 0, "a status was left set"


def stream_ptr():
    import torch
    return torch.cuda.current_stream().cuda_stream


def qkv(shape, dtype, cfg):
    return [inputs.normal_bits(shape, inputs.seed_for(cfg, t), dtype)
            for t in (inputs.TENSOR_Q, inputs.TENSOR_K, inputs.TENSOR_V)]


def oracle_prefill(oracle_mod, q, k, v, dtype, causal, scale, rows=None):
    f = [oracle_mod.bits_to_f64(x, dtype) for x in (q, k, v)]
    return oracle_mod.attention(*f, causal, scale, rows=rows, threads=G.THREADS)


# ------------------------------------------------------------ the plain calls
@pytest.mark.parametrize("causal", [False, True])
def test_fa_prefill_gpt2_b1(fa, oracle_mod, causal):
    # GPT-2-shaped prefill, B=1, H=12, N=2048, d=64, fp16 in and out, scale 1/8
    import torch
    B, H, N, d = 1, 12, 2048, 64
    q, k, v = qkv((B, H, N, d), "f16", CFG_GPT2)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))
    out = torch.full((B, H, N, d), float("nan"), dtype=torch.float16, device="cuda")
    rc = fa.fa_prefill(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B, H, N, d,
                       int(causal), 0.125, stream_ptr())
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    want = oracle_prefill(oracle_mod, q, k, v, "f16", causal, 0.125)
    G.assert_close(G.device_to_f64(out), want, "f16", "f16", f"fa_prefill causal={causal}")


@pytest.mark.parametrize("B,H", [(8, 12), (32, 14)])
def test_fa_decode_ragged(fa, oracle_mod, B, H):
    # ragged split-K decode: caches [B, H, 4096, 64] fp16, lengths uniform on [1, 4096]
    import torch
    L, d = 4096, 64
    q = inputs.normal_bits((B, H, 1, d), inputs.seed_for(CFG_DECODE, 0) + 7 * H, "f16")
    kc = inputs.normal_bits((B, H, L, d), inputs.seed_for(CFG_DECODE, 1) + 7 * H, "f16")
    vc = inputs.normal_bits((B, H, L, d), inputs.seed_for(CFG_DECODE, 2) + 7 * H, "f16")
    lens = inputs.seq_lens(inputs.seed_for(CFG_DECODE, inputs.TENSOR_SEQLEN) + 7 * B, B, L)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, kc, vc))
    ld = torch.from_numpy(lens).cuda()
    out = torch.full((B, H, 1, d), float("nan"), dtype=torch.float16, device="cuda")
    rc = fa.fa_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), ld.data_ptr(), out.data_ptr(),
                      B, H, L, d, 0.125, stream_ptr())
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    want = oracle_mod.decode(*(oracle_mod.bits_to_f64(x, "f16") for x in (q, kc, vc)), lens, 0.125,
                             threads=G.THREADS)
    G.assert_close(G.device_to_f64(out), want, "f16", "f16", f"fa_decode B={B} H={H}")
    assert fa.fa_device_status(False) == 0


def test_fa_prefill_ex_tiny_fp32_out_and_long_bf16(fa, oracle_mod):
    import torch
    # Tiny: B=1, H=2, N=128, d=64, fp16 in, fp32 out, full and causal
    q, k, v = qkv((1, 2, 128, 64), "f16", CFG_TINY)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))
    for causal in (0, 1):
        out = torch.empty((1, 2, 128, 64), dtype=torch.float32, device="cuda")
        rc = fa.fa_prefill_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), 1, 2, 128,
                              64, causal, 0.125, fa.FA_F16, fa.FA_F32, stream_ptr())
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        want = oracle_prefill(oracle_mod, q, k, v, "f16", causal, 0.125)
        G.assert_close(G.device_to_f64(out), want, "f16", "f32", f"tiny causal={causal}")
    # long dense: B=1, H=16, N=4096, d=128, bf16 in and out, sampled rows
    N, d = 4096, 128
    scale = float(np.float32(1.0 / np.sqrt(d)))
    q, k, v = qkv((1, 16, N, d), "bf16", CFG_LONG)
    qd, kd, vd = (G.bits_to_device(x, "bf16") for x in (q, k, v))
    out = torch.empty((1, 16, N, d), dtype=torch.bfloat16, device="cuda")
    rc = fa.fa_prefill_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), 1, 16, N, d, 0,
                          scale, fa.FA_BF16, fa.FA_BF16, stream_ptr())
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    rows = G.sample_rows(N, 41)
    want = oracle_prefill(oracle_mod, q, k, v, "bf16", False, scale, rows=rows)
    G.assert_close(G.device_to_f64(out)[:, :, rows], want, "bf16", "bf16", "long N=4096 via _ex")


def test_fa_decode_ex_with_caller_workspace(fa, oracle_mod):
    import torch
    B, H, L, d = 5, 3, 1500, 64
    q = inputs.normal_bits((B, H, 1, d), 901, "f16")
    kc = inputs.normal_bits((B, H, L, d), 902, "f16")
    vc = inputs.normal_bits((B, H, L, d), 903, "f16")
    lens = np.array([1500, 1, 64, 65, 999], dtype=np.int32)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, kc, vc))
    ld = torch.from_numpy(lens).cuda()
    splits = 9
    nbytes = fa.fa_decode_workspace_bytes(B, H, L, d, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H, 1, d), dtype=torch.float32, device="cuda")
    # one byte short is refused before anything is enqueued
    assert fa.fa_decode_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), ld.data_ptr(), out.data_ptr(),
                           B, H, L, d, 0.125, fa.FA_F16, fa.FA_F32, splits, ws.data_ptr(), nbytes - 1,
                           stream_ptr()) == fa.FA_ERR_WORKSPACE
    rc = fa.fa_decode_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), ld.data_ptr(), out.data_ptr(),
                         B, H, L, d, 0.125, fa.FA_F16, fa.FA_F32, splits, ws.data_ptr(), nbytes,
                         stream_ptr())
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    want = oracle_mod.decode(*(oracle_mod.bits_to_f64(x, "f16") for x in (q, kc, vc)), lens, 0.125)
    G.assert_close(G.device_to_f64(out), want, "f16", "f32", "fa_decode_ex workspace")


def test_split_choice_of_the_device(fa):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, H, L in [(1, 14, 4096), (32, 12, 4096), (3, 2, 1000)]:
        s = fa.fa_decode_choose_splits(B, H, L, 0)
        assert s == fa.fa_decode_choose_splits(B, H, L, -1) == fa.fa_decode_splits_for_sms(B, H, H, L, sms)
    assert fa.fa_decode_choose_splits(1, 1, 64, 1 << 20) == -fa.FA_ERR_CUDA  # no such device


# ------------------------------------------------------------ device status word
def test_packed_offsets_out_of_range_are_reported(fa, oracle_mod):
    import torch
    Hq, Hkv, d = 4, 2, 64
    total = 300
    q = inputs.normal_bits((total, Hq, d), 911, "f16")
    k = inputs.normal_bits((total, Hkv, d), 912, "f16")
    v = inputs.normal_bits((total, Hkv, d), 913, "f16")
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))

    def call(cu, max_len):
        cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
        out = torch.zeros((total, Hq, d), dtype=torch.float32, device="cuda")
        rc = fa.fa_prefill_varlen(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                                  cud.data_ptr(), cud.data_ptr(), len(cu) - 1, Hq, Hkv, total, total,
                                  max_len, max_len, d, 1, 0.125, fa.FA_F16, fa.FA_F32, 0, stream_ptr())
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        return G.device_to_f64(out)

    assert fa.fa_device_status(True) == 0
    got = call([0, 120, 300], 180)                       # valid: nothing reported
    assert fa.fa_device_status(False) == 0
    want = oracle_mod.attention_varlen(*(oracle_mod.bits_to_f64(x, "f16") for x in (q, k, v)),
                                       [0, 120, 300], [0, 120, 300], True, 0.125)
    G.assert_close(got, want, "f16", "f32", "packed batch")
    for cu, mx in [([0, 200, 150], 200),                 # decreasing offsets
                   ([0, 120, 400], 280),                 # past the end of the tensors
                   ([0, 120, 300], 100)]:                # a length above the stated maximum
        got = call(cu, mx)
        assert fa.fa_device_status(True) == fa.FA_ERR_SEQ_LEN, cu
        assert np.isfinite(got).all()
    assert fa.fa_device_status(False) == 0


def test_watchdog_fires_and_the_context_survives(fa, oracle_mod):
    import torch
    res = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    assert fa.fa_watchdog_selftest(1_000_000, res.data_ptr(), stream_ptr()) == fa.FA_OK   # 1 ms
    torch.cuda.synchronize()
    timed_out, aborted, t0_ns, t1_ns = (int(x) for x in res.cpu())
    assert timed_out == 1 and aborted == 1
    assert 1_000_000 <= t0_ns < 500_000_000
    # warp 1's own limit is 1.5 s: it returned on warp 0's abort flag instead
    assert 1_000_000 <= t1_ns < 500_000_000
    assert fa.fa_device_status(True) == fa.FA_ERR_WATCHDOG
    assert fa.fa_device_status(False) == 0
    # the next ordinary call runs normally and reports nothing
    q, k, v = qkv((1, 2, 256, 64), "f16", 920)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))
    out = fa.prefill(qd, kd, vd, causal=True, scale=0.125, out_dtype=torch.float32)
    torch.cuda.synchronize()
    G.assert_close(G.device_to_f64(out), oracle_prefill(oracle_mod, q, k, v, "f16", True, 0.125),
                   "f16", "f32", "prefill after the watchdog test")
    assert fa.fa_device_status(False) == 0
    # bad arguments are refused before any launch
    assert fa.fa_watchdog_selftest(10, res.data_ptr(), stream_ptr()) == fa.FA_ERR_SHAPE
    assert fa.fa_watchdog_selftest(1_000_000, res.data_ptr() + 4, stream_ptr()) == fa.FA_ERR_ALIGN
    assert fa.fa_watchdog_selftest(1_000_000, None, stream_ptr()) == fa.FA_ERR_NULL


# ------------------------------------------------------------ measurement helpers
def test_read_probe_reads_every_word(fa):
    import torch
    rng = np.random.default_rng(5)
    # sizes below one pass of the grid, and one with several unrolled passes and a tail
    for n in (16, 4096 + 16 * 7, 3 << 20, (64 << 20) + 48):
        host = rng.integers(0, 2 ** 32, size=n // 4, dtype=np.uint32)
        src = torch.from_numpy(host.view(np.int32)).cuda()
        x = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert fa.fa_read_probe(src.data_ptr(), n, x.data_ptr(), stream_ptr()) == fa.FA_OK
        torch.cuda.synchronize()
        want = np.bitwise_xor.reduce(host)
        assert int(x.cpu().numpy().view(np.uint32)[0]) == int(want), n
    assert fa.fa_read_probe(src.data_ptr(), 24, x.data_ptr(), stream_ptr()) == fa.FA_ERR_SHAPE
    assert fa.fa_read_probe(src.data_ptr() + 8, 32, x.data_ptr(), stream_ptr()) == fa.FA_ERR_ALIGN


def test_pool_counters_follow_an_allocating_call(fa):
    import torch
    rc, before = fa.fa_pool_stats(reset_high=True)
    assert rc == fa.FA_OK
    B, H, L, d = 4, 4, 2048, 64
    q, kc, vc = (torch.randn(s, device="cuda").half() for s in ((B, H, 1, d), (B, H, L, d), (B, H, L, d)))
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    fa.decode(q, kc, vc, lens, scale=0.125)          # workspace from the pool
    torch.cuda.synchronize()
    rc, after = fa.fa_pool_stats()
    assert rc == fa.FA_OK
    splits = fa.fa_decode_choose_splits(B, H, L, -1)
    assert after[3] >= fa.fa_decode_workspace_bytes(B, H, L, d, splits)  # in-use high-water mark
    assert after[2] == 0                                                # freed again
