"""The quantised record layout feeds the tensor-core fragments the codes they need.

include/pkv.h lays each code section out in the order the attention kernel's mma.sync
m16n8k16 A operands consume it.  This test takes records written by the oracle, reads each
lane's words of a 16-key group as the kernel does, widens them as the kernel does (Q8: one
prmt per f16 pair under the exponent 0x64; Q4 / Q2: bytes 1 and 3 moved down by one prmt,
then each field masked in place, value 1024 + 2^p u), and checks that A-fragment element
(register i, half e) of lane (g, c) decodes to the code of the key and dim the PTX fragment
layout assigns to it: A row g + 8 (i % 2), A column 2c + 8 (i // 2) + e, with K rows = keys
2g + r of the 16-key group and columns = dims of k-step ks, and V^T rows = dims of m-tile dm
and columns = keys in the order P^T arrives (2s for s < 8, 2(s - 8) + 1 otherwise).
"""
import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl


def _prmt(x, y, sel):
    src = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(src[(sel >> (4 * i)) & 0x7] << (8 * i) for i in range(4))


def _fpos(bits, step, half):
    return 0 if bits == 8 else (4 * half if bits == 4 else 4 * (step & 1) + 2 * half)


def _decode(h2, p, off):
    out = []
    for e in range(2):
        v = (h2 >> (16 * e)) & 0xFFFF
        assert v >> 10 == 0x19                      # f16 exponent of 1024
        m = v & 0x3FF
        assert m % (1 << p) == 0
        out.append(m // (1 << p) - off)
    return out


def _fragments(bits, cw, step, is_v):
    """The kernel's A registers for k-step (K) or dim m-tile (V) `step`, with field positions."""
    if bits == 8:
        w0, w1 = cw[2 * step], cw[2 * step + 1]
        a = [_prmt(w0, 0x64646464, 0x4240), _prmt(w1, 0x64646464, 0x4240),
             _prmt(w0, 0x64646464, 0x4341), _prmt(w1, 0x64646464, 0x4341)]
        return a, [0, 0, 0, 0]
    lo = cw[step] if bits == 4 else cw[step >> 1]
    hi = _prmt(lo, 0, 0x3311)
    f = 0x000F000F if bits == 4 else 0x00030003
    p0, p1 = _fpos(bits, step, 0), _fpos(bits, step, 1)
    m0, m1 = f << p0, f << p1
    E = 0x64006400
    if not is_v:   # byte = row half r, field = column half h
        return [(lo & m0) | E, (hi & m0) | E, (lo & m1) | E, (hi & m1) | E], [p0, p0, p1, p1]
    return [(lo & m0) | E, (lo & m1) | E, (hi & m0) | E, (hi & m1) | E], [p0, p1, p0, p1]


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("D,BS", [(64, 16), (64, 32), (128, 16), (128, 32)])
def test_record_codes_land_in_fragment_order(oracle_mod, bits, D, BS):
    rng = np.random.default_rng(100 * bits + D + BS)
    rec = oracle_mod.new_qpool(1, 1, BS, D, bits)
    rows = wl.f32_to_bf16_bits(rng.standard_normal((BS, 1, D)).astype(np.float32))
    oracle_mod.paged_kv_append_quant(rec, BS, D, bits, np.array([[0]], np.int32), np.zeros(1, np.int32),
                                     np.array([0, BS], np.int32), rows, rows)
    codes = np.array([oracle_mod.kv_quantize_row(rows[t, 0], bits)[0] for t in range(BS)])
    raw = rec[0, 0]
    C = BS * D * bits // 8
    NW = D * bits // 64                      # words per lane per 16-key group
    off = 1 << (bits - 1)

    def lane_words(section, group, lane):
        base = section + group * NW * 4 * 32
        if bits == 2:                        # one contiguous run per lane
            starts = [base + lane * NW * 4 + 4 * k for k in range(NW)]
        else:                                # 16-byte units interleaved across the warp
            starts = [base + ((k // 4) * 32 + lane) * 16 + 4 * (k % 4) for k in range(NW)]
        return [int.from_bytes(raw[s:s + 4].tobytes(), "little") for s in starts]

    for group in range(BS // 16):
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            for is_v in (False, True):
                cw = lane_words(C if is_v else 0, group, lane)
                for step in range(D // 16):
                    regs, pos = _fragments(bits, cw, step, is_v)
                    for i in range(4):
                        vals = _decode(regs[i], pos[i], off)
                        row, col0 = g + 8 * (i % 2), 2 * c + 8 * (i // 2)
                        for e in range(2):
                            col = col0 + e
                            if is_v:
                                dim, key = 16 * step + row, 16 * group + (2 * col if col < 8 else 2 * (col - 8) + 1)
                            else:
                                key, dim = 16 * group + 2 * (row % 8) + row // 8, 16 * step + col
                            assert vals[e] == codes[key, dim], (is_v, lane, step, i, e)
