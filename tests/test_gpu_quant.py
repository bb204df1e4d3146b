"""GPU parity of the quantised KV path (Q8 / Q4 / Q2 records) against the float64 oracle.

TensorSharp "高级功能", section "内存优化", the KV block codec item.  Bars: the
quantising append bit-exact (codes and scales, byte for byte); attention max-abs
<= 2e-2 and mean-abs <= 2e-3 against the oracle's attention over the same records;
batch-vs-solo, window-row-vs-decode and NaN-in-unused-slots bit-identical on the GPU
(TensorFold article, section "先记住一条铁律").
"""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import assert_close_to_oracle, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BITS = [8, 4, 2]


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _status_ok(pkv):
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0, f"device status {rc}, bits {bits:#x}"


def _dev(b, rec, layer=0):
    return dict(rec=dev(rec), block_tables=dev(b.block_tables), context_lens_old=dev(b.context_lens_old),
                context_lens=dev(b.context_lens), new_starts=dev(b.new_starts),
                k_new=dev_bf16(b.k_new[layer]), v_new=dev_bf16(b.v_new[layer]),
                q_starts=dev(b.q_starts), q=dev_bf16(b.q[layer]),
                sinks=None if b.sinks is None else dev(b.sinks))


def _gpu_qstep(pkv, b, rec, bits, layer=0, out_dtype=None, g=None):
    g = g or _dev(b, rec, layer)
    B, D = b.block_size, b.head_dim
    if b.new_starts[-1] > 0:
        pkv.paged_kv_append_quant(g["rec"], B, D, bits, g["block_tables"], g["context_lens_old"],
                                  g["new_starts"], g["k_new"], g["v_new"])
    out = pkv.paged_attention_forward_quant(
        g["rec"], B, D, bits, g["q"], g["q_starts"], g["block_tables"], g["context_lens"],
        max_context_len=max(1, b.max_context_len), max_q_rows_per_seq=max(1, b.max_q_rows_per_seq),
        sinks=g["sinks"], causal=b.causal, out_dtype=out_dtype or torch.bfloat16)
    torch.cuda.synchronize()
    return g, out


def _oracle_qstep(b, rec, bits, layer=0):
    r = rec.copy()
    if b.new_starts[-1] > 0:
        oracle.paged_kv_append_quant(r, b.block_size, b.head_dim, bits, b.block_tables, b.context_lens_old,
                                     b.new_starts, b.k_new[layer], b.v_new[layer])
    ref = oracle.paged_attention_quant(r, b.block_size, b.head_dim, bits, b.q[layer], b.q_starts,
                                       b.block_tables, b.context_lens, sinks=b.sinks, causal=b.causal)
    return r, ref


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("name,filler", [("tiny_decode", "random"), ("spec_verify", "nan"),
                                         ("cb_mix", "random"), ("window_d64_b32", "nan")])
def test_append_quant_bit_exact(pkv, bits, name, filler):
    if name == "window_d64_b32":
        lens = np.array([5, 32, 33, 70, 100])
        W = np.array([5, 16, 2, 16, 9])
        b = wl.build_batch(9, name=name, lens=lens, n_new=W, q_rows=W, num_q_heads=8, num_kv_heads=2,
                           head_dim=64, block_size=32, causal=True, filler=filler)
    else:
        b = wl.make_workload(name, seed=0, filler=filler, num_seqs=4 if name != "tiny_decode" else None)
    b.k_new[0][0, 0, :] = 0                   # a zero row: scale 0, every code 0
    rec = wl.random_records(1, b, bits, filler=filler)[0]
    g, _ = _gpu_qstep(pkv, b, rec, bits)
    r = rec.copy()
    oracle.paged_kv_append_quant(r, b.block_size, b.head_dim, bits, b.block_tables, b.context_lens_old,
                                 b.new_starts, b.k_new[0], b.v_new[0])
    got = g["rec"].cpu().numpy()
    assert np.array_equal(got, r), f"{int((got != r).sum())} record bytes differ"
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("name,seed,filler", [("tiny_decode", 0, "nan"), ("tiny_decode", 1, "random"),
                                              ("cb_mix", 0, "random"), ("spec_verify", 0, "nan"),
                                              ("sinks_scale", 0, "random")])
def test_attention_quant_matches_oracle(pkv, bits, name, seed, filler):
    b = wl.make_workload(name, seed=seed, filler=filler)
    rec = wl.random_records(seed + 10, b, bits, filler=filler)[0]
    _, out = _gpu_qstep(pkv, b, rec, bits)
    _, ref = _oracle_qstep(b, rec, bits)
    mx, mean = assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"q{bits} {name}/{seed}")
    print(f"q{bits} {name} seed {seed}: max-abs {mx:.2e} mean-abs {mean:.2e}")
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("d,bs", [(64, 16), (64, 32), (128, 16), (128, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_quant_ragged_lengths_all_variants(pkv, bits, d, bs, causal):
    # every block and split boundary (quantised splits are 1024 keys) and one past it
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1023, 1024, 1025, 2048, 2049, 3073])
    W = np.array([1, 1, 3, 2, 16, 1, 5, 16, 1, 7, 16, 1, 16, 3, 9, 12]) if causal else np.ones(len(lens), np.int64)
    W = np.minimum(W, lens)
    b = wl.build_batch(31 + d + bs + bits, name="ragged", lens=lens, n_new=W, q_rows=W, num_q_heads=16,
                       num_kv_heads=2, head_dim=d, block_size=bs, causal=causal, with_sinks=causal,
                       filler="nan")
    rec = wl.random_records(bits + d + bs, b, bits, filler="nan")[0]
    _, out = _gpu_qstep(pkv, b, rec, bits)
    _, ref = _oracle_qstep(b, rec, bits)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"q{bits} d{d} bs{bs} causal{causal}")
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
def test_quant_wide_dynamic_range_queries(pkv, bits):
    # q entries spanning 2^-24 .. 2^8 (the kernel scales some dims by 2^-fpos before rounding
    # to f16, so its tiniest entries go subnormal), an all-zero row and a single-spike row
    lens = np.array([300, 1200, 77])
    W = np.array([1, 4, 2])
    b = wl.build_batch(61 + bits, name="qrange", lens=lens, n_new=W, q_rows=W, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, block_size=16, causal=True, with_sinks=True)
    rng = np.random.default_rng(62 + bits)
    q = rng.standard_normal(b.q[0].shape) * 2.0 ** rng.uniform(-24, 8, size=b.q[0].shape)
    q[0] = 0.0
    q[1] = 0.0
    q[1, :, 5] = 37.0
    b.q[0] = wl.f32_to_bf16_bits(q.astype(np.float32))
    rec = wl.random_records(70 + bits, b, bits)[0]
    _, out = _gpu_qstep(pkv, b, rec, bits)
    _, ref = _oracle_qstep(b, rec, bits)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"q{bits} wide-range q")
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("name", ["cb_mix", "spec_verify"])
def test_quant_batch_vs_solo_bit_identical(pkv, bits, name):
    b = wl.make_workload(name, seed=4)
    rec = wl.random_records(4, b, bits)[0]
    g, out = _gpu_qstep(pkv, b, rec, bits)
    full = host_bits(out)
    for s in range(0, b.num_seqs, 3):
        sub = wl.select_seqs(b, [s])
        one = pkv.paged_attention_forward_quant(
            g["rec"], b.block_size, b.head_dim, bits, dev_bf16(sub.q[0]), dev(sub.q_starts),
            dev(sub.block_tables), dev(sub.context_lens), max_context_len=max(1, sub.max_context_len),
            max_q_rows_per_seq=max(1, sub.max_q_rows_per_seq), causal=b.causal)
        torch.cuda.synchronize()
        r0, r1 = b.q_starts[s], b.q_starts[s + 1]
        assert np.array_equal(host_bits(one), full[r0:r1]), f"sequence {s} differs alone"
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
def test_quant_window_rows_equal_single_row_decodes(pkv, bits):
    b = wl.make_workload("spec_verify", seed=5)
    rec = wl.random_records(5, b, bits)[0]
    g, out = _gpu_qstep(pkv, b, rec, bits)
    full = host_bits(out)
    for s in range(0, b.num_seqs, 3):
        W, L = int(b.q_starts[s + 1] - b.q_starts[s]), int(b.context_lens[s])
        for w in range(W):
            r = int(b.q_starts[s]) + w
            one = pkv.paged_attention_forward_quant(
                g["rec"], b.block_size, b.head_dim, bits, g["q"][r:r + 1].contiguous(),
                dev(np.array([0, 1], np.int32)), g["block_tables"][s:s + 1].contiguous(),
                dev(np.array([L - W + w + 1], np.int32)), max_context_len=L, max_q_rows_per_seq=1, causal=False)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(one)[0], full[r]), f"seq {s} row {w}"


@pytest.mark.parametrize("bits", BITS)
def test_quant_window_rows_straddling_split_boundaries(pkv, bits):
    # causal windows of 16 rows whose rows end on both sides of a 512-, 1024- and 2048-key
    # boundary: every row equals the one-row decode over its own keys, bit for bit
    lens = np.array([520, 1030, 2056, 1031, 3080])
    W = np.array([16, 16, 16, 9, 16])
    b = wl.build_batch(90 + bits, name="straddle", lens=lens, n_new=W, q_rows=W, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=16, causal=True, filler="nan")
    rec = wl.random_records(91 + bits, b, bits, filler="nan")[0]
    g, out = _gpu_qstep(pkv, b, rec, bits)
    full = host_bits(out)
    _, ref = _oracle_qstep(b, rec, bits)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"q{bits} straddling windows")
    for s in range(b.num_seqs):
        w_s, L = int(W[s]), int(b.context_lens[s])
        for w in range(w_s):
            r = int(b.q_starts[s]) + w
            one = pkv.paged_attention_forward_quant(
                g["rec"], b.block_size, b.head_dim, bits, g["q"][r:r + 1].contiguous(),
                dev(np.array([0, 1], np.int32)), g["block_tables"][s:s + 1].contiguous(),
                dev(np.array([L - w_s + w + 1], np.int32)), max_context_len=L, max_q_rows_per_seq=1, causal=False)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(one)[0], full[r]), f"seq {s} row {w}"
    _status_ok(pkv)


@pytest.mark.parametrize("bits", BITS)
def test_quant_nan_scales_in_unused_slots_change_nothing(pkv, bits):
    b = wl.make_workload("spec_verify", seed=8, num_seqs=6)
    ra = wl.random_records(8, b, bits, filler="random")[0]
    rn = wl.random_records(8, b, bits, filler="nan")[0]
    _, out_a = _gpu_qstep(pkv, b, ra, bits)
    _, out_n = _gpu_qstep(pkv, b, rn, bits)
    assert np.array_equal(host_bits(out_a), host_bits(out_n))


def test_quant_host_side_argument_errors(pkv):
    b = wl.make_workload("tiny_decode", seed=0)
    rec = wl.random_records(0, b, 8)[0]
    g = _dev(b, rec)
    lib = pkv.lib()
    pool = pkv._qpool(g["rec"], b.block_size, b.head_dim, 8)
    pool.bits = 5
    import ctypes
    rc = lib.paged_attention_forward_quant(ctypes.byref(pool), pkv._dptr(g["q"]), pkv._dptr(g["q_starts"]),
                                           pkv._dptr(g["block_tables"]), b.block_tables.shape[1],
                                           pkv._dptr(g["context_lens"]), b.num_seqs, b.total_q_rows, 1024, 1,
                                           b.num_q_heads, None, None, 0, 0.0, pkv._dptr(g["q"]), 0,
                                           pkv._dptr(g["rec"]), 1 << 20, None)
    assert rc == -3
    pool.bits = 8
    pool.records = g["rec"].data_ptr() + 8
    rc = lib.paged_kv_append_quant(ctypes.byref(pool), pkv._dptr(g["block_tables"]), b.block_tables.shape[1],
                                   pkv._dptr(g["context_lens_old"]), pkv._dptr(g["new_starts"]),
                                   pkv._dptr(g["k_new"]), pkv._dptr(g["v_new"]), b.num_seqs, 4, None)
    assert rc == -7
    with pytest.raises(ValueError):
        pkv._qpool(g["rec"], b.block_size, b.head_dim, 4)   # record size of another codec
