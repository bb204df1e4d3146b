"""Oracle pins for quantised KV blocks (Q8 / Q4 / Q2 codec, record layout, attention).

TensorSharp "高级功能", section "内存优化", the KV block codec item: blocks are
compressed in place to 8, 4 or 2 bits per value at a small accuracy cost.  The codec
(per-row symmetric integer codes with one float32 scale) and the record layout
are this library's reading; they are pinned by hand-worked examples, the
rounding error bound, a layout bijection, and by exactly representable data on
which quantised attention must equal the (separately pinned) bf16 attention.
"""
import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl

QMAX = {8: 127, 4: 7, 2: 1}


def bf(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_quantize_worked_examples(oracle_mod):
    # amax 127 -> scale exactly 1; codes are x rounded half to even
    codes, scale = oracle_mod.kv_quantize_row(bf([127, -63.5, 0, 1, 0.5, -0.5, 1.5, 2.5, -2.5, 126.5]), 8)
    assert scale == 1.0
    assert codes.tolist() == [127, -64, 0, 1, 0, 0, 2, 2, -2, 126]
    # 4 bits: amax 7 -> scale 1
    codes, scale = oracle_mod.kv_quantize_row(bf([7, -3.5, 2.5, 0.375, -7, 1.5]), 4)
    assert scale == 1.0
    assert codes.tolist() == [7, -4, 2, 0, -7, 2]
    # amax 2 -> scale = fl32(2/7) = 2/7 + (3/7) 2^-25, slightly above 2/7.  Then
    # -1 / scale = -(3.5 - 1.56e-7), which float32 rounds to -(3.5 - 2^-22) (the nearer
    # neighbour), so the code is -3, not the -4 a real-number tie would give: the codec's
    # decisions are float32 ones.  0.5 / scale -> 1.75 - 8e-8 -> 2.
    codes, scale = oracle_mod.kv_quantize_row(bf([2, 0.5, -1, 0]), 4)
    assert scale == np.float32(2) / np.float32(7)
    assert codes.tolist() == [7, 2, -3, 0]
    # 2 bits: Q = 1, amax 3 -> scale 3; x / 3 rounds to -1, 0 or 1 (+-0.5 ties go to 0)
    codes, scale = oracle_mod.kv_quantize_row(bf([3, -1.5, 1.5, 2, -3, 1, -2, 0]), 2)
    assert scale == 3.0
    assert codes.tolist() == [1, 0, 0, 1, -1, 0, -1, 0]
    # a zero row: scale 0, every code 0
    codes, scale = oracle_mod.kv_quantize_row(bf([0, -0.0, 0, 0]), 8)
    assert scale == 0.0 and not codes.any()


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantize_error_bound_and_range(oracle_mod, bits):
    rng = np.random.default_rng(bits)
    Q = QMAX[bits]
    for trial in range(200):
        d = 128 if trial % 2 else 64
        x = bf(rng.standard_normal(d) * 10.0 ** rng.uniform(-3, 3))
        xf = wl.bf16_bits_to_f32(x).astype(np.float64)
        codes, scale = oracle_mod.kv_quantize_row(x, bits)
        amax = np.abs(xf).max()
        assert np.all(np.abs(codes) <= Q)
        assert np.abs(codes).max() == Q                       # the largest value maps to +-Q
        assert abs(float(scale) - amax / Q) <= amax / Q * 2 ** -23
        err = np.abs(codes * np.float64(scale) - xf)
        # round to nearest, up to the float32 rounding of x / scale (|x / scale| <= Q)
        assert np.all(err <= np.float64(scale) * (0.5 + Q * 2 ** -23))


@pytest.mark.parametrize("bits,D,BS", [(8, 128, 16), (8, 64, 32), (4, 128, 16), (4, 64, 32),
                                        (2, 128, 16), (2, 64, 16), (2, 64, 32)])
def test_record_layout_is_a_bijection(oracle_mod, bits, D, BS):
    C = BS * D * bits // 8
    assert oracle_mod.qrecord_bytes(BS, D, bits) == 2 * C + 8 * BS
    for sec in (0, 1):
        seen = {}
        for t in range(BS):
            for i in range(D):
                off, sh = oracle_mod.qcode_offset(sec, t, i, D, BS, bits)
                assert sec * C <= off < (sec + 1) * C
                assert (off, sh) not in seen
                seen[(off, sh)] = t
        assert len(seen) == BS * D
        # every byte holds codes of one slot only (tokens append independently)
        by_byte = {}
        for (off, sh), t in seen.items():
            by_byte.setdefault(off, set()).add(t)
        assert len(by_byte) == C and all(len(v) == 1 for v in by_byte.values())


def test_record_layout_worked_offsets(oracle_mod):
    # slot 3, dim 37, head_dim 128, block 16, worked by hand from the documented formula
    assert oracle_mod.qcode_offset(0, 3, 37, 128, 16, 8) == (614, 0)
    assert oracle_mod.qcode_offset(1, 3, 37, 128, 16, 8) == (2048 + 835, 0)
    assert oracle_mod.qcode_offset(0, 3, 37, 128, 16, 4) == (107, 0)
    assert oracle_mod.qcode_offset(1, 3, 37, 128, 16, 4) == (1024 + 331, 0)
    assert oracle_mod.qcode_offset(0, 1, 0, 128, 16, 8) == (4, 0)       # key parity 1, column parity 0
    assert oracle_mod.qcode_offset(0, 0, 1, 128, 16, 8) == (2, 0)       # key parity 0, column parity 1
    assert oracle_mod.qcode_offset(0, 1, 0, 128, 16, 4) == (1, 0)       # bit 8
    assert oracle_mod.qcode_offset(0, 0, 1, 128, 16, 4) == (2, 0)       # bit 16
    assert oracle_mod.qcode_offset(0, 0, 8, 128, 16, 4) == (0, 4)       # h = 1: high nibble
    assert oracle_mod.qcode_offset(1, 0, 8, 128, 16, 4) == (1024, 4)    # r = 1: high nibble
    # 2 bits (units of D/8 = 16 bytes): K slot 3 (g 1, r 1), dim 37 (j 2, c 2, h 0, e 1) -> u 6,
    # word 96 + 4, bit 8 + 0 + 16 = 24; V slot 3 (m 9: h 1, c 0, e 1), dim 37 (dm 2, g 5,
    # r 0) -> u 20, word 512 + 320 + 4, bit 8 + 16 = 24
    assert oracle_mod.qcode_offset(0, 3, 37, 128, 16, 2) == (103, 0)
    assert oracle_mod.qcode_offset(1, 3, 37, 128, 16, 2) == (512 + 327, 0)
    assert oracle_mod.qcode_offset(0, 1, 0, 128, 16, 2) == (1, 0)       # r = 1, e = 0: byte 1
    assert oracle_mod.qcode_offset(0, 0, 1, 128, 16, 2) == (2, 0)       # r = 0, e = 1: byte 2
    assert oracle_mod.qcode_offset(0, 0, 8, 128, 16, 2) == (0, 2)       # h = 1
    assert oracle_mod.qcode_offset(0, 0, 16, 128, 16, 2) == (0, 4)      # j = 1: second k-step
    assert oracle_mod.qcode_offset(1, 0, 8, 128, 16, 2) == (512, 2)     # r = 1
    assert oracle_mod.qcode_offset(1, 1, 0, 128, 16, 2) == (513, 0)     # slot 1: m 8, h 1, e 0
    assert oracle_mod.qcode_offset(1, 2, 0, 128, 16, 2) == (514, 0)     # slot 2: m 1, h 0, e 1
    assert oracle_mod.qcode_offset(1, 0, 16, 128, 16, 2) == (512, 4)    # dm = 1
    assert oracle_mod.qcode_offset(0, 16, 0, 64, 32, 2) == (32 * 8, 0)  # head_dim 64: 8-byte units


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_append_writes_only_its_slots(oracle_mod, bits):
    rng = np.random.default_rng(20 + bits)
    H, D, BS, nb = 2, 64, 16, 6
    rec = oracle_mod.new_qpool(nb, H, BS, D, bits)
    rec[...] = rng.integers(0, 256, size=rec.shape, dtype=np.uint8)
    before = rec.copy()
    # two sequences: s0 appends 3 tokens at positions 14..16 (crossing into a new block), s1 one at 5
    bt = np.array([[4, 1, -1], [2, -1, -1]], np.int32)
    old = np.array([14, 5], np.int32)
    ns = np.array([0, 3, 4], np.int32)
    kn = bf(rng.standard_normal((4, H, D)))
    vn = bf(rng.standard_normal((4, H, D)))
    oracle_mod.paged_kv_append_quant(rec, BS, D, bits, bt, old, ns, kn, vn)
    k, v = oracle_mod.qpool_dequant(rec, BS, D, bits)
    k0, v0 = oracle_mod.qpool_dequant(before, BS, D, bits)
    written = {(4, 14): 0, (4, 15): 1, (1, 0): 2, (2, 5): 3}
    for (blk, slot), row in written.items():
        for h in range(H):
            for pool, new in ((k, kn), (v, vn)):
                codes, scale = oracle_mod.kv_quantize_row(new[row, h], bits)
                assert np.array_equal(pool[blk, h, slot], codes * np.float64(scale))
    mask = np.ones((nb, H, BS), bool)
    for (blk, slot) in written:
        mask[blk, :, slot] = False
    # untouched slots are byte-for-byte the filler (whose scales may decode to NaN)
    assert np.array_equal(k[mask], k0[mask], equal_nan=True) and np.array_equal(v[mask], v0[mask], equal_nan=True)


def _exact_batch(rng, bits, S=3, H=2, Hq=4, D=64, BS=16):
    """Pools whose rows are integers in [-Q, Q] times a power of two, each with a +-Q entry:
    the codec represents them exactly."""
    Q = QMAX[bits]
    lens = np.array([37, 16, 70][:S], np.int32)
    nblk = (lens + BS - 1) // BS
    nb = int(nblk.sum()) + 2
    perm = rng.permutation(nb)
    bt = -np.ones((S, int(nblk.max())), np.int32)
    k = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    vals = rng.integers(-Q, Q + 1, size=(2, nb, H, BS, D)).astype(np.float64)
    vals[..., 0] = Q * np.where(rng.random((2, nb, H, BS)) < 0.5, -1, 1)
    pw = 2.0 ** rng.integers(-6, 3, size=(2, nb, H, BS, 1))
    kv = bf(vals * pw)
    return lens, bt, kv, nb


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantised_attention_equals_bf16_attention_on_exact_data(oracle_mod, bits):
    rng = np.random.default_rng(30 + bits)
    H, Hq, D, BS = 2, 4, 64, 16
    lens, bt, kv, nb = _exact_batch(rng, bits, H=H, Hq=Hq, D=D, BS=BS)
    kp, vp = kv[0], kv[1]
    # fill the record pool through the quantising append of every cached token
    rec = oracle_mod.new_qpool(nb, H, BS, D, bits)
    S = len(lens)
    rows = [np.stack([kp[bt[s, t // BS], :, t % BS] for t in range(lens[s])]) for s in range(S)]
    vrows = [np.stack([vp[bt[s, t // BS], :, t % BS] for t in range(lens[s])]) for s in range(S)]
    ns = np.zeros(S + 1, np.int32)
    ns[1:] = np.cumsum(lens)
    oracle_mod.paged_kv_append_quant(rec, BS, D, bits, bt, np.zeros(S, np.int32), ns,
                                     np.concatenate(rows), np.concatenate(vrows))
    qs = np.array([0, 1, 3, 4], np.int32)
    q = bf(rng.standard_normal((4, Hq, D)))
    sinks = rng.standard_normal(Hq).astype(np.float32)
    for causal, sk in ((False, None), (True, sinks)):
        ref = oracle_mod.paged_attention(kp, vp, q, qs, bt, lens, sinks=sk, causal=causal)
        got = oracle_mod.paged_attention_quant(rec, BS, D, bits, q, qs, bt, lens, sinks=sk, causal=causal)
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("bits,bound", [(8, 0.05), (4, 0.6), (2, 3.5)])
def test_quantised_attention_accuracy_cost(oracle_mod, bits, bound):
    # random N(0,1) K/V: the codec's cost on the output (loose, informative bounds; ternary
    # 2-bit codes with one scale per row keep only a Gaussian row's largest entries, so
    # their cost is of the order of the output itself)
    rng = np.random.default_rng(40 + bits)
    H, Hq, D, BS, S, L = 2, 8, 128, 16, 2, 300
    nb = S * ((L + BS - 1) // BS)
    bt = np.arange(nb, dtype=np.int32).reshape(S, -1)
    lens = np.full(S, L, np.int32)
    kp = bf(rng.standard_normal((nb, H, BS, D)))
    vp = bf(rng.standard_normal((nb, H, BS, D)))
    rec = oracle_mod.new_qpool(nb, H, BS, D, bits)
    ns = np.array([0, L, 2 * L], np.int32)
    rows_k = np.concatenate([np.stack([kp[bt[s, t // BS], :, t % BS] for t in range(L)]) for s in range(S)])
    rows_v = np.concatenate([np.stack([vp[bt[s, t // BS], :, t % BS] for t in range(L)]) for s in range(S)])
    oracle_mod.paged_kv_append_quant(rec, BS, D, bits, bt, np.zeros(S, np.int32), ns, rows_k, rows_v)
    q = bf(rng.standard_normal((S, Hq, D)) * 2)
    qs = np.arange(S + 1, dtype=np.int32)
    ref = oracle_mod.paged_attention(kp, vp, q, qs, bt, lens)
    got = oracle_mod.paged_attention_quant(rec, BS, D, bits, q, qs, bt, lens)
    assert np.abs(got - ref).max() < bound
