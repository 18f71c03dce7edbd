"""GPU parity of the prefill kernel against the fp64 oracle (through the C ABI).

Workloads follow the five configurations of the target (seeded N(0,1) data;
seeds 0xFA000000 + 16 * config + tensor): Tiny, GPT-2-shaped, long dense
d=128, and the causal stress case with 1% outlier keys x20.  Small shapes are
checked element by element in full; the full-size ones on sampled rows
(every head, tile-boundary rows plus seeded rows) -- rows are independent, so
a sampled row is an exact check of that row.
"""
import numpy as np
import pytest

from attention_forward_prefill_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

CFG_TINY, CFG_GPT2, CFG_LONG, CFG_DECODE, CFG_STRESS = 0, 1, 2, 3, 4


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


def make_qkv(shape, dtype, cfg, outliers=False):
    q = inputs.normal_bits(shape, inputs.seed_for(cfg, inputs.TENSOR_Q), dtype)
    if outliers:
        k, rows = inputs.keys_with_outliers(shape, inputs.seed_for(cfg, inputs.TENSOR_K),
                                            inputs.seed_for(cfg, inputs.TENSOR_OUTLIER), dtype)
    else:
        k, rows = inputs.normal_bits(shape, inputs.seed_for(cfg, inputs.TENSOR_K), dtype), None
    v = inputs.normal_bits(shape, inputs.seed_for(cfg, inputs.TENSOR_V), dtype)
    return q, k, v, rows


def run_prefill(fa, q, k, v, dtype, causal, scale, out_dtype, flags=0):
    import torch
    qd, kd, vd = (G.bits_to_device(x, dtype) for x in (q, k, v))
    out = fa.prefill(qd, kd, vd, causal=causal, scale=scale, out_dtype=G.torch_dtype(out_dtype),
                     flags=flags)
    torch.cuda.synchronize()
    return out


def oracle_rows(oracle_mod, q, k, v, dtype, causal, scale, rows=None, b_chunk=1):
    """Oracle output [B, H, R, d] from the same bits, one batch element at a time."""
    B = q.shape[0]
    outs = []
    for b0 in range(0, B, b_chunk):
        sl = slice(b0, b0 + b_chunk)
        qf, kf, vf = (oracle_mod.bits_to_f64(x[sl], dtype) for x in (q, k, v))
        outs.append(oracle_mod.attention(qf, kf, vf, causal, scale, rows=rows, threads=G.THREADS))
    return np.concatenate(outs, axis=0)


def check(fa, oracle_mod, shape, dtype, out_dtype, causal, scale, cfg, rows=None,
          outliers=False, extra_rows_fn=None):
    q, k, v, orows = make_qkv(shape, dtype, cfg, outliers)
    out = run_prefill(fa, q, k, v, dtype, causal, scale, out_dtype)
    got = G.device_to_f64(out)
    if rows is not None and extra_rows_fn is not None:
        rows = np.unique(np.concatenate([rows, extra_rows_fn(orows)]))
    want = oracle_rows(oracle_mod, q, k, v, dtype, causal, scale, rows=rows)
    if rows is not None:
        got = got[:, :, rows]
    return G.assert_close(got, want, dtype, out_dtype, f"prefill {shape} {dtype}->{out_dtype} "
                          f"causal={causal}")


# ------------------------------------------------------------ the five configs
@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(fa, oracle_mod, causal):
    check(fa, oracle_mod, (1, 2, 128, 64), "f16", "f32", causal, 0.125, CFG_TINY)


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_config_b1_full(fa, oracle_mod, causal):
    check(fa, oracle_mod, (1, 12, 2048, 64), "f16", "f16", causal, 0.125, CFG_GPT2)


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_config_b4_sampled(fa, oracle_mod, causal):
    check(fa, oracle_mod, (4, 12, 2048, 64), "f16", "f16", causal, 0.125, CFG_GPT2,
          rows=G.sample_rows(2048, 11))


def check_bf16_and_strict_fp32(fa, oracle_mod, shape, causal, cfg, rows, outliers=False,
                               extra_rows_fn=None):
    """One bf16 problem run twice: bf16 output against 8e-3 + half an output
    ulp, and fp32 output against the plain 8e-3 (the output rounding then
    cannot hide a kernel error), both on the same oracle rows."""
    scale = float(np.float32(1.0 / np.sqrt(shape[-1])))
    q, k, v, orows = make_qkv(shape, "bf16", cfg, outliers)
    if extra_rows_fn is not None:
        rows = np.unique(np.concatenate([rows, extra_rows_fn(orows)]))
    want = oracle_rows(oracle_mod, q, k, v, "bf16", causal, scale, rows=rows)
    got = G.device_to_f64(run_prefill(fa, q, k, v, "bf16", causal, scale, "bf16"))[:, :, rows]
    G.assert_close(got, want, "bf16", "bf16", f"prefill {shape} bf16 causal={causal}")
    got32 = G.device_to_f64(run_prefill(fa, q, k, v, "bf16", causal, scale, "f32"))[:, :, rows]
    err = float(np.abs(got32 - want).max())
    assert err <= 8e-3, f"prefill {shape} fp32 output: max abs err {err:.3e} > 8e-3"


@pytest.mark.parametrize("N", [4096, 8192, 16384])
def test_long_dense_config_sampled(fa, oracle_mod, N):
    check_bf16_and_strict_fp32(fa, oracle_mod, (1, 16, N, 128), False, CFG_LONG,
                               G.sample_rows(N, N))


def test_stress_config_sampled(fa, oracle_mod):
    N = 8192

    def outlier_neighbourhood(orows):
        r = np.unique(orows[:, :4].reshape(-1))[:8]
        return np.clip(np.concatenate([r, r + 1]), 0, N - 1)

    check_bf16_and_strict_fp32(fa, oracle_mod, (8, 32, N, 128), True, CFG_STRESS,
                               G.sample_rows(N, 5), outliers=True,
                               extra_rows_fn=outlier_neighbourhood)


# ------------------------------------------------------------ edge shapes
@pytest.mark.parametrize("N", [1, 2, 127, 129, 255, 256, 257, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths_full_check(fa, oracle_mod, N, d, causal):
    dtype = "bf16" if d == 128 else "f16"
    check(fa, oracle_mod, (2, 3, N, d), dtype, "f32", causal, 1.0 / np.sqrt(d), 100 + N)


@pytest.mark.parametrize("in_dtype,out_dtype", [("f16", "bf16"), ("bf16", "f16"),
                                                ("bf16", "f32"), ("f16", "f16")])
def test_dtype_combinations(fa, oracle_mod, in_dtype, out_dtype):
    check(fa, oracle_mod, (1, 4, 384, 64), in_dtype, out_dtype, True, 0.125, 200)


# ------------------------------------------------------------ special cases
def test_zero_scale_gives_mean_of_visible_values(fa, oracle_mod):
    q, k, v, _ = make_qkv((1, 2, 300, 64), "f16", 201)
    got = G.device_to_f64(run_prefill(fa, q, k, v, "f16", True, 0.0, "f32"))
    vf = oracle_mod.bits_to_f64(v, "f16")
    want = np.cumsum(vf, axis=2) / np.arange(1, 301)[None, None, :, None]
    assert np.abs(got - want).max() <= 2e-3


def test_negative_scale(fa, oracle_mod):
    check(fa, oracle_mod, (1, 2, 333, 64), "f16", "f32", False, -0.2, 202)
    check(fa, oracle_mod, (1, 2, 333, 128), "bf16", "f32", True, -0.1, 203)


def test_causal_row_zero_is_exactly_first_value_row(fa):
    q, k, v, _ = make_qkv((2, 4, 512, 128), "bf16", 204)
    got = run_prefill(fa, q, k, v, "bf16", True, 0.0884, "f32").float().cpu().numpy()
    vf = (v.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(got[:, :, 0], vf[:, :, 0])


def test_identical_value_rows(fa):
    import torch
    shape = (1, 3, 700, 64)
    q, k, _, _ = make_qkv(shape, "f16", 205)
    row = inputs.normal_bits((64,), 7, "f16")
    v = np.broadcast_to(row, shape).copy()
    got = G.device_to_f64(run_prefill(fa, q, k, v, "f16", False, 0.3, "f32"))
    want = row.view(np.float16).astype(np.float64)
    assert np.abs(got - want).max() <= 2e-3


# ------------------------------------------------------------ determinism
@pytest.mark.parametrize("causal", [True, False])
def test_run_to_run_bit_identical(fa, causal):
    import torch
    q, k, v, _ = make_qkv((4, 12, 2048, 64), "f16", CFG_GPT2)
    outs = [run_prefill(fa, q, k, v, "f16", causal, 0.125, "f16") for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("shape", [(1, 24, 8192, 64), (1, 3, 1000, 64), (2, 5, 4100, 128)])
def test_units_cut_across_ctas(fa, oracle_mod, shape):
    # When the last wave of 256-row units would leave most SMs idle, the
    # non-causal work is spread over all SMs in equal step ranges, so a unit
    # can be cut between CTAs and merged afterwards (768 and 170 units here on
    # ~150 SMs); the small shape keeps the unit-per-CTA schedule.
    B, H, N, d = shape
    dtype = "bf16" if d == 128 else "f16"
    check(fa, oracle_mod, shape, dtype, "f32", False, 1.0 / np.sqrt(d), 210 + N,
          rows=G.sample_rows(N, 7) if N > 2048 else None)


@pytest.mark.parametrize("N,d", [(2048, 64), (1000, 128), (4096, 128)])
def test_causal_tile_skip_is_bit_identical(fa, N, d):
    import torch
    dtype = "bf16" if d == 128 else "f16"
    q, k, v, _ = make_qkv((2, 4, N, d), dtype, 206)
    # same schedule for both (skipping changes unit costs, which may change the
    # library's choice between the two schedules and with it the summation order)
    units = fa.FA_FLAG_SCHEDULE_UNITS
    a = run_prefill(fa, q, k, v, dtype, True, 1.0 / np.sqrt(d), dtype, flags=units)
    b = run_prefill(fa, q, k, v, dtype, True, 1.0 / np.sqrt(d), dtype,
                    flags=units | fa.FA_FLAG_NO_CAUSAL_SKIP)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_host_tensors_end_to_end(fa, oracle_mod):
    import torch
    q, k, v, _ = make_qkv((1, 2, 256, 64), "f16", 207)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16).copy()).view(torch.float16).pin_memory()
                  for x in (q, k, v))
    out = fa.prefill(qh, kh, vh, causal=True, scale=0.125, out_dtype=torch.float32)
    assert not out.is_cuda
    want = oracle_rows(oracle_mod, q, k, v, "f16", True, 0.125)
    assert np.abs(out.numpy().astype(np.float64) - want).max() <= 2e-3


# ------------------------------------------------------------ very long sequences
@pytest.mark.parametrize("shape,causal", [((1, 1, 300_000, 64), True), ((1, 2, 65_536, 128), False)])
def test_very_long_sequences_sampled(fa, oracle_mod, shape, causal):
    # 300K rows: more query blocks than the stream-K step table holds (1024),
    # so the unit schedule runs; 64K rows dense: stream-K with a 256-entry table.
    # Row indices and TMA coordinates run far past 2^16.
    B, H, N, d = shape
    dtype = "bf16" if d == 128 else "f16"
    rows = G.sample_rows(N, 19, extra=(65_535, 65_536, 131_071, 262_143, 299_999))
    check(fa, oracle_mod, shape, dtype, "f32", causal, 1.0 / np.sqrt(d), 230, rows=rows)
