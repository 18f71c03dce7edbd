"""GPU parity of the general prefill forms against the fp64 oracle (C ABI):
chunked prompts (Nq != Nk, queries aligned to the last keys), grouped key /
value heads, packed variable-length batches, and the stream-K schedule on
causal work (forced by flag, including more CTAs than key-tile steps).
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
    assert torch.cuda.get_device_capability() == (10, 3), "libfa_gb300 targets sm_103a"
    build.build()
    binding.load()
    assert binding.fa_device_status(True) == 0
    yield binding
    assert binding.fa_device_status(False) == 0, "a kernel watchdog fired"


def gen(shape, seed, dtype):
    return inputs.normal_bits(shape, seed, dtype)


def run_dense(fa, q, k, v, dtype, causal, scale, out_dtype, flags=0):
    import torch
    qd, kd, vd = (G.bits_to_device(x, dtype) for x in (q, k, v))
    out = fa.prefill(qd, kd, vd, causal=causal, scale=scale, out_dtype=G.torch_dtype(out_dtype),
                     flags=flags)
    torch.cuda.synchronize()
    return G.device_to_f64(out)


def oracle_dense(oracle_mod, q, k, v, dtype, causal, scale, rows=None):
    qf, kf, vf = (oracle_mod.bits_to_f64(x, dtype) for x in (q, k, v))
    return oracle_mod.attention(qf, kf, vf, causal, scale, rows=rows, threads=G.THREADS)


def check_dense(fa, oracle_mod, B, Hq, Hkv, Nq, Nk, d, causal, seed, out_dtype="f32", flags=0,
                rows=None):
    dtype = "bf16" if d == 128 else "f16"
    q = gen((B, Hq, Nq, d), seed, dtype)
    k = gen((B, Hkv, Nk, d), seed + 1, dtype)
    v = gen((B, Hkv, Nk, d), seed + 2, dtype)
    scale = 1.0 / np.sqrt(d)
    got = run_dense(fa, q, k, v, dtype, causal, scale, out_dtype, flags)
    want = oracle_dense(oracle_mod, q, k, v, dtype, causal, scale, rows)
    if rows is not None:
        got = got[:, :, rows]
    G.assert_close(got, want, dtype, out_dtype,
                   f"prefill B={B} Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal={causal}")
    return got


# ------------------------------------------------------------ chunked prompts
@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1, 777), (129, 513), (256, 4096), (1000, 1000)])
@pytest.mark.parametrize("causal", [True, False])
def test_chunk_over_longer_keys(fa, oracle_mod, Nq, Nk, causal):
    check_dense(fa, oracle_mod, 1, 4, 4, Nq, Nk, 64, causal, 400 + Nq)
    check_dense(fa, oracle_mod, 1, 2, 2, Nq, Nk, 128, causal, 500 + Nq)


@pytest.mark.parametrize("Nq,Nk", [(500, 200), (300, 1), (257, 129)])
def test_more_queries_than_keys(fa, oracle_mod, Nq, Nk):
    # causal: the first Nq - Nk rows see no key and must come back as zeros
    got = check_dense(fa, oracle_mod, 2, 2, 2, Nq, Nk, 64, True, 600 + Nq)
    assert np.array_equal(got[:, :, : Nq - Nk], np.zeros_like(got[:, :, : Nq - Nk]))


# ------------------------------------------------------------ grouped heads
@pytest.mark.parametrize("Hq,Hkv", [(14, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_kv_heads(fa, oracle_mod, Hq, Hkv, causal):
    check_dense(fa, oracle_mod, 2, Hq, Hkv, 700, 700, 64, causal, 700 + Hq)
    check_dense(fa, oracle_mod, 1, Hq, Hkv, 384, 640, 128, causal, 800 + Hq)


def test_grouped_heads_equal_repeated_heads_on_the_gpu(fa):
    # the kernel's own result with repeated K/V heads must match bit for bit
    import torch
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 64
    q = G.bits_to_device(gen((B, Hq, N, d), 901, "f16"), "f16")
    k = G.bits_to_device(gen((B, Hkv, N, d), 902, "f16"), "f16")
    v = G.bits_to_device(gen((B, Hkv, N, d), 903, "f16"), "f16")
    a = fa.prefill(q, k, v, causal=True, scale=0.125)
    b = fa.prefill(q, k.repeat_interleave(4, dim=1).contiguous(),
                   v.repeat_interleave(4, dim=1).contiguous(), causal=True, scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------ packed batches
def pack(seqs_q, seqs_k, Hq, Hkv, d, dtype, seed):
    cu_q = np.concatenate([[0], np.cumsum(seqs_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seqs_k)]).astype(np.int32)
    q = gen((max(int(cu_q[-1]), 1), Hq, d), seed, dtype)[: cu_q[-1]]
    k = gen((max(int(cu_k[-1]), 1), Hkv, d), seed + 1, dtype)[: cu_k[-1]]
    v = gen((max(int(cu_k[-1]), 1), Hkv, d), seed + 2, dtype)[: cu_k[-1]]
    return q, k, v, cu_q, cu_k


def run_varlen(fa, q, k, v, cu_q, cu_k, dtype, causal, scale, out_dtype="f32"):
    import torch
    qd, kd, vd = (G.bits_to_device(np.ascontiguousarray(x), dtype) for x in (q, k, v))
    cq = torch.from_numpy(cu_q).cuda()
    ck = torch.from_numpy(cu_k).cuda()
    mq = int(np.max(np.diff(cu_q)))
    mk = int(np.max(np.diff(cu_k)))
    out = fa.prefill_varlen(qd, kd, vd, cq, ck, mq, mk, causal=causal, scale=scale,
                            out_dtype=G.torch_dtype(out_dtype))
    torch.cuda.synchronize()
    return G.device_to_f64(out)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens", [
    ([1, 130, 257, 0, 600], None),                 # self-attention, ragged, one empty
    ([100, 1, 300, 64], [612, 77, 300, 2000]),     # chunks over longer caches
    ([200, 50], [0, 50]),                          # a sequence with no keys
])
def test_packed_variable_length_batch(fa, oracle_mod, d, causal, lens):
    lq, lk = lens
    lk = lq if lk is None else lk
    dtype = "bf16" if d == 128 else "f16"
    Hq, Hkv = 4, 2
    q, k, v, cu_q, cu_k = pack(lq, lk, Hq, Hkv, d, dtype, 1000 + d + sum(lq))
    scale = 1.0 / np.sqrt(d)
    got = run_varlen(fa, q, k, v, cu_q, cu_k, dtype, causal, scale)
    want = oracle_mod.attention_varlen(oracle_mod.bits_to_f64(q, dtype), oracle_mod.bits_to_f64(k, dtype),
                                       oracle_mod.bits_to_f64(v, dtype), cu_q, cu_k, causal, scale,
                                       threads=G.THREADS)
    G.assert_close(got, want, dtype, "f32", f"varlen d={d} causal={causal} lens={lq}/{lk}")


def test_packed_batch_equals_dense_batch_when_lengths_agree(fa):
    import torch
    B, H, N, d = 3, 4, 300, 64
    q = gen((B, H, N, d), 1100, "f16")
    k = gen((B, H, N, d), 1101, "f16")
    v = gen((B, H, N, d), 1102, "f16")
    dense = run_dense(fa, q, k, v, "f16", True, 0.125, "f16")
    tq, tk, tv = (np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(B * N, H, d)) for x in (q, k, v))
    cu = (np.arange(B + 1) * N).astype(np.int32)
    packed = run_varlen(fa, tq, tk, tv, cu, cu, "f16", True, 0.125, "f16")
    assert np.array_equal(packed.reshape(B, N, H, d).transpose(0, 2, 1, 3), dense)
    del torch


@pytest.mark.parametrize("d,dtype", [(64, "f16"), (128, "bf16")])
@pytest.mark.parametrize("causal", [True, False])
def test_packed_batch_over_several_rounds_equals_its_sequences_alone(fa, oracle_mod, d, dtype, causal):
    # 21 sequences of 0 to 1500 tokens, 8 query heads over 2 key/value heads:
    # about 1000 units, several rounds on 152 SMs, dealt heaviest (sequence,
    # block) class first from an order computed on the device.  Every unit is
    # whole in one CTA, so each sequence's rows must be bit-identical to the same
    # sequence run alone as a dense batch under the unit schedule.
    rng = np.random.default_rng(1300 + d + causal)
    lens = [int(x) for x in rng.integers(1, 1500, 20)] + [0]
    rng.shuffle(lens)
    Hq, Hkv = 8, 2
    q, k, v, cu_q, cu_k = pack(lens, lens, Hq, Hkv, d, dtype, 1310 + d)
    scale = 1.0 / np.sqrt(d)
    got = run_varlen(fa, q, k, v, cu_q, cu_k, dtype, causal, scale)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(int(cu_q[b]), int(cu_q[b + 1]))
        qs, ks, vs = (np.ascontiguousarray(x[sl].transpose(1, 0, 2)[None]) for x in (q, k, v))
        alone = run_dense(fa, qs, ks, vs, dtype, causal, scale, "f32", flags=fa.FA_FLAG_SCHEDULE_UNITS)
        assert np.array_equal(got[sl].transpose(1, 0, 2)[None], alone), f"sequence {b} ({n} tokens)"
    b = int(np.argmax(lens))
    sl = slice(int(cu_q[b]), int(cu_q[b + 1]))
    qs, ks, vs = (np.ascontiguousarray(x[sl].transpose(1, 0, 2)[None]) for x in (q, k, v))
    rows = G.sample_rows(lens[b], 5)
    want = oracle_dense(oracle_mod, qs, ks, vs, dtype, causal, scale, rows=rows)
    G.assert_close(got[sl].transpose(1, 0, 2)[None][:, :, rows], want, dtype, "f32",
                   f"packed sequence {b} d={d} causal={causal}")


# ------------------------------------------------------------ stream-K, causal
@pytest.mark.parametrize("shape", [(1, 12, 12, 2048, 2048, 64), (2, 3, 3, 1000, 1000, 128),
                                   (1, 4, 2, 700, 1500, 64), (1, 2, 2, 300, 300, 64)])
def test_causal_stream_k_schedule(fa, oracle_mod, shape):
    # forced stream-K on causal work: units of unequal cost cut between CTAs,
    # a query tile whose keys end before a piece starts, and (last shape) more
    # CTAs than key-tile steps
    B, Hq, Hkv, Nq, Nk, d = shape
    rows = G.sample_rows(Nq, 17) if Nq > 1024 else None
    sk = check_dense(fa, oracle_mod, B, Hq, Hkv, Nq, Nk, d, True, 1200 + Nq,
                     flags=fa.FA_FLAG_SCHEDULE_STREAM_K, rows=rows)
    un = check_dense(fa, oracle_mod, B, Hq, Hkv, Nq, Nk, d, True, 1200 + Nq,
                     flags=fa.FA_FLAG_SCHEDULE_UNITS, rows=rows)
    assert np.abs(sk - un).max() <= 4e-3


@pytest.mark.parametrize("causal", [False, True])
def test_stream_k_unit_cut_into_many_pieces(fa, oracle_mod, causal):
    # a 256-query chunk over 16384 keys with two heads: the schedule cuts each of
    # the two units over 76 CTAs, so the fixup's piece list takes several warp
    # ballots and merges 76 partials per row
    _, info, items = fa.fa_prefill_plan(1, 2, 256, 16384, causal, 0, 0)  # this device's SMs
    if info[0] and info[1] == 152:
        assert [it[2] - it[1] + 1 for it in items] == [76, 76]
    check_dense(fa, oracle_mod, 1, 2, 2, 256, 16384, 128, causal, 1500 + causal, rows=G.sample_rows(256, 19))


def test_stream_k_is_bit_identical_run_to_run(fa):
    import torch
    B, H, N, d = 1, 12, 2048, 64
    q, k, v = (G.bits_to_device(gen((B, H, N, d), 1300 + i, "f16"), "f16") for i in range(3))
    outs = [fa.prefill(q, k, v, causal=True, scale=0.125, flags=fa.FA_FLAG_SCHEDULE_STREAM_K)
            for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_stream_k_non_causal_with_idle_ctas(fa, oracle_mod):
    check_dense(fa, oracle_mod, 1, 2, 2, 300, 300, 64, False, 1400,
                flags=fa.FA_FLAG_SCHEDULE_STREAM_K)
    check_dense(fa, oracle_mod, 1, 3, 1, 200, 900, 128, False, 1401,
                flags=fa.FA_FLAG_SCHEDULE_STREAM_K)


def test_many_small_units(fa, oracle_mod):
    # 64 x 32 heads of 64 causal rows: 2048 one-tile units, about 13 rounds of
    # the unit schedule per CTA, each unit's second query tile empty
    check_dense(fa, oracle_mod, 64, 32, 32, 64, 64, 64, True, 4100, rows=None)


def test_grouped_heads_under_stream_k_with_a_ragged_tail(fa, oracle_mod):
    # 4 x 40 query heads over 8 key/value heads, N = 1000 (a ragged last tile):
    # dense and non-causal, so the library may cut units between CTAs
    _, info, _ = fa.fa_prefill_plan(4, 40, 1000, 1000, 0, 0, 0)
    check_dense(fa, oracle_mod, 4, 40, 8, 1000, 1000, 128, False, 4200,
                rows=G.sample_rows(1000, 3))
    check_dense(fa, oracle_mod, 4, 40, 8, 1000, 1000, 128, False, 4200,
                flags=fa.FA_FLAG_SCHEDULE_STREAM_K, rows=G.sample_rows(1000, 3))
