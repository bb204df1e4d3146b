"""GPU parity of the index-list gather against the float64 oracle.

TensorSharp "高级功能", the DeepSeek V4 executor item ([ring | top-k] keys through an
index-gather).  Bars: max-abs <= 2e-2 and mean-abs <= 2e-3 against the oracle; a row
in a batch equals the row alone, bit for bit; a list naming every key in order equals
paged_attention_forward, bit for bit (same tiles, same arithmetic).
"""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import assert_close_to_oracle, dev, dev_bf16, gpu_batch, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _status_ok(pkv):
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0, f"device status {rc}, bits {bits:#x}"


def _run(pkv, b, g, k=0):
    out = pkv.paged_attention_forward_gather(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                             g["context_lens"], dev(b.key_idx[k]), dev(b.key_counts[k]),
                                             sinks=g["sinks"])
    torch.cuda.synchronize()
    return out


def _ref(b, k=0):
    return oracle.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                         b.context_lens, b.key_idx[k], b.key_counts[k], sinks=b.sinks)


@pytest.mark.parametrize("seed", [0, 1])
def test_sparse_gather_matches_oracle(pkv, seed):
    b = wl.make_workload("sparse_gather", seed=seed, num_seqs=24, filler="nan")
    g = gpu_batch(b)
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    kp, vp = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle.paged_kv_append(kp, vp, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    b.k_pool, b.v_pool = kp[None], vp[None]
    for k in range(2):
        got = _run(pkv, b, g, k).float().cpu().numpy()
        mx, mean = assert_close_to_oracle(got, _ref(b, k), what=f"gather seed {seed} set {k}")
        print(f"gather seed {seed} set {k}: max-abs {mx:.2e} mean-abs {mean:.2e}")
    _status_ok(pkv)


@pytest.mark.parametrize("d,bs,G", [(64, 16, 8), (64, 32, 4), (128, 16, 5), (128, 32, 16)])
def test_ragged_lists_and_shapes(pkv, d, bs, G):
    lens = np.array([1, 15, 17, 512, 513, 1300, 3000])
    Hkv = 2
    b = wl.build_batch(40 + d + bs + G, name="gl", lens=lens, n_new=np.zeros(len(lens), np.int64),
                       q_rows=np.array([1, 2, 1, 3, 1, 2, 1]), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                       head_dim=d, block_size=bs, causal=False, with_sinks=True, filler="nan")
    rng = np.random.default_rng(d + bs + G)
    R = b.total_q_rows
    width = 1100
    idx = np.full((1, R, width), -1, np.int32)
    cnt = np.zeros((1, R), np.int32)
    row_seq = np.searchsorted(b.q_starts, np.arange(R), side="right") - 1
    for r in range(R):
        L = int(b.context_lens[row_seq[r]])
        n = [0, 1, 16, 17, 511, 512, 513, 1100][r % 8]
        n = min(n, 2 * L)
        lst = rng.integers(0, L, n).astype(np.int32)          # repeats allowed
        idx[0, r, :n] = lst
        cnt[0, r] = n
    b.key_idx, b.key_counts = idx, cnt
    g = gpu_batch(b)
    got = _run(pkv, b, g).float().cpu().numpy()
    assert_close_to_oracle(got, _ref(b), what=f"d{d} bs{bs} G{G}")
    _status_ok(pkv)


def test_full_in_order_list_equals_paged_attention(pkv):
    b = wl.make_workload("tiny_decode", seed=3)
    g = gpu_batch(b)
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    dense = pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                        g["context_lens"], max_context_len=b.max_context_len, max_q_rows_per_seq=1)
    L = b.context_lens
    idx = np.full((1, b.total_q_rows, int(L.max())), -1, np.int32)
    for r in range(b.total_q_rows):
        idx[0, r, :L[r]] = np.arange(L[r])
    b.key_idx, b.key_counts = idx, L.astype(np.int32)[None]
    got = _run(pkv, b, g)
    assert np.array_equal(host_bits(got), host_bits(dense))


def test_batch_vs_solo_bit_identical(pkv):
    b = wl.make_workload("sparse_gather", seed=4, num_seqs=16)
    g = gpu_batch(b)
    full = host_bits(_run(pkv, b, g))
    for s in range(0, b.num_seqs, 3):
        sub = wl.select_seqs(b, [s])
        gs = dict(g, q=dev_bf16(sub.q[0]), q_starts=dev(sub.q_starts), block_tables=dev(sub.block_tables),
                  context_lens=dev(sub.context_lens))
        one = host_bits(_run(pkv, sub, gs))
        assert np.array_equal(one, full[b.q_starts[s]:b.q_starts[s + 1]]), f"sequence {s}"


def test_out_of_range_position_is_flagged(pkv):
    b = wl.make_workload("tiny_decode", seed=5)
    g = gpu_batch(b)
    idx = np.zeros((1, b.total_q_rows, 4), np.int32)
    idx[0, 2, 1] = int(b.context_lens[2]) + 5
    b.key_idx, b.key_counts = idx, np.full((1, b.total_q_rows), 4, np.int32)
    out = _run(pkv, b, g)
    assert torch.isfinite(out.float()).all()
    rc, bits = pkv.device_status()
    assert rc == -5 and bits == 2                              # PKV_DEV_TABLE_OVERRUN
    _run(pkv, b, g)                                            # the context stays usable
    pkv.device_status()
