"""GPU parity of split-K decode against the fp64 oracle (through the C ABI).

Ragged-decode configuration: B in {1, 8, 32}, H in {14, 12}, d = 64, fp16
caches [B, H, 4096, 64], per-sequence lengths uniform on [1, 4096], scale 1/8.
Every output is checked (decode is cheap for the oracle).  Also: decode of
token t equals row t of causal prefill, invariance over every split count,
bit-identical reruns for a fixed split, lengths at chunk edges.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
CFG_DECODE = 3


@pytest.fixture(scope="module")
def fa():
    import torch
    from attention_forward_prefill_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3), "libfa_gb300 targets sm_103a"
    build.build()
    binding.load()
    return binding


def make_decode(B, H, L, d, dtype, cfg, lens=None):
    q = inputs.normal_bits((B, H, 1, d), inputs.seed_for(cfg, inputs.TENSOR_Q) + 1000 * H, dtype)
    kc = inputs.normal_bits((B, H, L, d), inputs.seed_for(cfg, inputs.TENSOR_K) + 1000 * H, dtype)
    vc = inputs.normal_bits((B, H, L, d), inputs.seed_for(cfg, inputs.TENSOR_V) + 1000 * H, dtype)
    if lens is None:
        lens = inputs.seq_lens(inputs.seed_for(cfg, inputs.TENSOR_SEQLEN) + B, B, L)
    return q, kc, vc, np.asarray(lens, dtype=np.int32)


def run_decode(fa, q, kc, vc, lens, dtype, scale, out_dtype="f16", num_splits=0, workspace=None):
    import torch
    out = fa.decode(G.bits_to_device(q, dtype), G.bits_to_device(kc, dtype),
                    G.bits_to_device(vc, dtype), torch.from_numpy(lens).cuda(), scale=scale,
                    out_dtype=G.torch_dtype(out_dtype), num_splits=num_splits,
                    workspace=workspace)
    torch.cuda.synchronize()
    return out


def oracle_decode(oracle_mod, q, kc, vc, lens, dtype, scale):
    return oracle_mod.decode(oracle_mod.bits_to_f64(q, dtype), oracle_mod.bits_to_f64(kc, dtype),
                             oracle_mod.bits_to_f64(vc, dtype), lens, scale, threads=G.THREADS)


@pytest.mark.parametrize("B", [1, 8, 32])
@pytest.mark.parametrize("H", [14, 12])
def test_ragged_decode_config(fa, oracle_mod, B, H):
    q, kc, vc, lens = make_decode(B, H, 4096, 64, "f16", CFG_DECODE)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    G.assert_close(got, want, "f16", "f16", f"decode B={B} H={H}")


def test_lengths_at_chunk_edges(fa, oracle_mod):
    L, B, H = 4096, 11, 3
    splits = fa.fa_decode_choose_splits(B, H, L, -1)
    chunk = fa.fa_decode_chunk_len(L, splits)
    lens = [1, 2, chunk - 1, chunk, chunk + 1, 2 * chunk, 2 * chunk + 1, L - 1, L, 63, 65]
    lens = [min(max(x, 1), L) for x in lens]
    q, kc, vc, lens = make_decode(B, H, L, 64, "f16", 300, lens)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32"))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    G.assert_close(got, want, "f16", "f32", "decode chunk edges")


def test_every_split_count_agrees(fa, oracle_mod):
    L, B, H = 1000, 3, 2
    q, kc, vc, lens = make_decode(B, H, L, 64, "f16", 301, [1000, 517, 64])
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    max_splits = (L + 63) // 64
    first = None
    for s in range(1, max_splits + 1):
        got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32", num_splits=s))
        G.assert_close(got, want, "f16", "f32", f"decode splits={s}")
        if first is None:
            first = got
        assert np.abs(got - first).max() <= 2e-3


def test_more_than_32_splits(fa, oracle_mod):
    # the merge kernel reads (m, l) 32 splits to a batch: past 32 splits it takes
    # a second batch of lanes.  At 64 splits the chunks are 64 rows, so these
    # lengths have 64, 40 and 33 splits with keys; 32 splits stay in one batch.
    L, B, H = 4096, 3, 2
    assert fa.fa_decode_chunk_len(L, 64) == 64
    q, kc, vc, lens = make_decode(B, H, L, 64, "f16", 302, [4096, 2500, 2049])
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    for s in (32, 64):
        got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32", num_splits=s))
        G.assert_close(got, want, "f16", "f32", f"decode splits={s}")


def test_fixed_split_is_bit_identical_and_workspace_paths_agree(fa):
    import torch
    B, H, L = 8, 14, 4096
    q, kc, vc, lens = make_decode(B, H, L, 64, "f16", CFG_DECODE)
    a = run_decode(fa, q, kc, vc, lens, "f16", 0.125)
    b = run_decode(fa, q, kc, vc, lens, "f16", 0.125)
    splits = fa.fa_decode_choose_splits(B, H, L, -1)
    nbytes = fa.fa_decode_workspace_bytes(B, H, L, 64, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    c = run_decode(fa, q, kc, vc, lens, "f16", 0.125, workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_decode_of_token_t_equals_causal_prefill_row_t(fa):
    import torch
    B, H, N, d = 2, 12, 1024, 64
    q = inputs.normal_bits((B, H, N, d), 11, "f16")
    k = inputs.normal_bits((B, H, N, d), 12, "f16")
    v = inputs.normal_bits((B, H, N, d), 13, "f16")
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, k, v))
    pre = fa.prefill(qd, kd, vd, causal=True, scale=0.125, out_dtype=torch.float32)
    for t in [0, 1, 63, 64, 500, N - 1]:
        lens = torch.full((B,), t + 1, dtype=torch.int32, device="cuda")
        dec = fa.decode(qd[:, :, t:t + 1].contiguous(), kd, vd, lens, scale=0.125,
                        out_dtype=torch.float32)
        torch.cuda.synchronize()
        diff = (dec[:, :, 0] - pre[:, :, t]).abs().max().item()
        assert diff <= 2e-3, (t, diff)


def test_length_clamping_and_zero_length(fa, oracle_mod):
    B, H, L = 4, 2, 300
    q, kc, vc, _ = make_decode(B, H, L, 64, "f16", 302, [1, 1, 1, 1])
    assert fa.fa_device_status(True) == 0
    # a zero length is legal (a zero row) and is not reported
    lens = np.array([0, 300, 17, 0], dtype=np.int32)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32"))
    assert fa.fa_device_status(False) == 0
    # lengths outside [0, max_len] are clamped, and the clamp is reported once
    lens = np.array([0, 300, 5000, -7], dtype=np.int32)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32"))
    want = oracle_decode(oracle_mod, q, kc, vc, np.clip(lens, 0, L), "f16", 0.125)
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert np.array_equal(got[3], np.zeros_like(got[3]))
    G.assert_close(got, want, "f16", "f32", "decode clamped lengths")
    assert fa.fa_device_status(True) == fa.FA_ERR_SEQ_LEN
    assert fa.fa_device_status(False) == 0


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "bf16"), (128, "f16")])
def test_other_head_dims_and_dtypes(fa, oracle_mod, d, dtype):
    B, H, L = 5, 4, 2000
    q, kc, vc, lens = make_decode(B, H, L, d, dtype, 303)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, dtype, 1.0 / np.sqrt(d), "f32"))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, dtype, 1.0 / np.sqrt(d))
    G.assert_close(got, want, dtype, "f32", f"decode d={d} {dtype}")


# ------------------------------------------------------------ grouped cache heads
def make_gqa(B, Hq, Hkv, L, d, dtype, seed, lens=None):
    q = inputs.normal_bits((B, Hq, 1, d), seed, dtype)
    kc = inputs.normal_bits((B, Hkv, L, d), seed + 1, dtype)
    vc = inputs.normal_bits((B, Hkv, L, d), seed + 2, dtype)
    if lens is None:
        lens = inputs.seq_lens(seed + 3, B, L)
    return q, kc, vc, np.asarray(lens, dtype=np.int32)


@pytest.mark.parametrize("B", [1, 8, 32])
def test_grouped_decode_qwen_shape(fa, oracle_mod, B):
    # Qwen2.5-0.5B-like attention: 14 query heads over 2 cache heads, d = 64
    q, kc, vc, lens = make_gqa(B, 14, 2, 4096, 64, "f16", 1500 + B)
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    G.assert_close(got, want, "f16", "f16", f"grouped decode B={B}")


@pytest.mark.parametrize("Hq,Hkv,d,dtype", [(8, 1, 64, "f16"), (4, 2, 128, "bf16"), (32, 2, 64, "f16"),
                                            (12, 1, 128, "bf16"), (6, 2, 64, "bf16")])
def test_grouped_decode_group_sizes(fa, oracle_mod, Hq, Hkv, d, dtype):
    q, kc, vc, lens = make_gqa(3, Hq, Hkv, 2000, d, dtype, 1600 + Hq, [2000, 1, 777])
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, dtype, 1.0 / np.sqrt(d), "f32"))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, dtype, 1.0 / np.sqrt(d))
    G.assert_close(got, want, dtype, "f32", f"grouped decode Hq={Hq} Hkv={Hkv} d={d}")


def test_grouped_decode_equals_repeated_caches_bitwise(fa):
    # the grouped kernel does each head's arithmetic in the plain kernel's order
    import torch
    B, Hq, Hkv, L = 4, 14, 2, 3000
    q, kc, vc, lens = make_gqa(B, Hq, Hkv, L, 64, "f16", 1700)
    qd, kd, vd = (G.bits_to_device(x, "f16") for x in (q, kc, vc))
    ld = torch.from_numpy(lens).cuda()
    a = fa.decode(qd, kd, vd, ld, scale=0.125, num_splits=6)
    b = fa.decode(qd, kd.repeat_interleave(7, dim=1).contiguous(),
                  vd.repeat_interleave(7, dim=1).contiguous(), ld, scale=0.125, num_splits=6)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_grouped_decode_equals_one_row_chunk_prefill(fa):
    import torch
    B, Hq, Hkv, N, d = 2, 14, 2, 1500, 64
    q = G.bits_to_device(inputs.normal_bits((B, Hq, N, d), 1800, "f16"), "f16")
    k = G.bits_to_device(inputs.normal_bits((B, Hkv, N, d), 1801, "f16"), "f16")
    v = G.bits_to_device(inputs.normal_bits((B, Hkv, N, d), 1802, "f16"), "f16")
    for t in [0, 127, 128, 999, N - 1]:
        lens = torch.full((B,), t + 1, dtype=torch.int32, device="cuda")
        qt = q[:, :, t:t + 1].contiguous()
        dec = fa.decode(qt, k, v, lens, scale=0.125, out_dtype=torch.float32)
        pre = fa.prefill(qt, k[:, :, : t + 1].contiguous(), v[:, :, : t + 1].contiguous(), causal=True,
                         scale=0.125, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert (dec - pre).abs().max().item() <= 2e-3, t


def test_very_long_cache_many_splits(fa, oracle_mod):
    # 262,144 cache rows: the automatic choice keeps chunks at most 512 rows, so
    # 512 splits and the merge walks 16 batches of 32 (m, l) lanes
    B, H, L = 2, 2, 262_144
    q, kc, vc, _ = make_decode(B, H, L, 64, "f16", 310, [1, 1])
    lens = np.array([L, 100_003], dtype=np.int32)
    splits = fa.fa_decode_choose_splits(B, H, L, -1)
    assert splits >= 512
    got = G.device_to_f64(run_decode(fa, q, kc, vc, lens, "f16", 0.125, "f32"))
    want = oracle_decode(oracle_mod, q, kc, vc, lens, "f16", 0.125)
    G.assert_close(got, want, "f16", "f32", "decode over 262144 rows")
