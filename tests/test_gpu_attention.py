"""GPU parity of paged append + paged attention against the float64 oracle.

Bars: append bit-exact; attention max-abs <= 2e-2 and mean-abs <= 2e-3 against the
oracle; batch-vs-solo, window-row-vs-decode, block permutation, shared-vs-duplicated
prefix and NaN-filled unused slots bit-identical on the GPU itself (TensorFold article,
section "先记住一条铁律": a row computed in a batch or a verify window equals the row
computed alone).
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


def _gpu_step(pkv, b, layer=0, out_dtype=None, g=None, **kw):
    g = g or gpu_batch(b, layer)
    if b.new_starts[-1] > 0:
        pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"],
                            g["new_starts"], g["k_new"], g["v_new"])
    out = pkv.paged_attention_forward(
        g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"], g["context_lens"],
        max_context_len=max(1, b.max_context_len), max_q_rows_per_seq=max(1, b.max_q_rows_per_seq),
        sinks=g["sinks"], causal=b.causal, out_dtype=out_dtype or torch.bfloat16, **kw)
    torch.cuda.synchronize()
    return g, out


def _oracle_step(b, layer=0, **kw):
    k, v = b.k_pool[layer].copy(), b.v_pool[layer].copy()
    if b.new_starts[-1] > 0:
        oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts,
                               b.k_new[layer], b.v_new[layer])
    ref = oracle.paged_attention(k, v, b.q[layer], b.q_starts, b.block_tables, b.context_lens,
                                 sinks=b.sinks, causal=b.causal, **kw)
    return k, v, ref


def _attn_only(pkv, g, b, tables=None, lens=None, q=None, q_starts=None, k_pool=None, v_pool=None,
               max_ctx=None, max_rows=None, **kw):
    out = pkv.paged_attention_forward(
        g["k_pool"] if k_pool is None else k_pool, g["v_pool"] if v_pool is None else v_pool,
        g["q"] if q is None else q, g["q_starts"] if q_starts is None else q_starts,
        g["block_tables"] if tables is None else tables, g["context_lens"] if lens is None else lens,
        max_context_len=max_ctx or max(1, b.max_context_len),
        max_q_rows_per_seq=max_rows or max(1, b.max_q_rows_per_seq),
        sinks=g["sinks"], causal=b.causal, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,filler", [("tiny_decode", "random"), ("tiny_decode", "nan"),
                                         ("cb_mix", "random"), ("spec_verify", "random")])
def test_append_bit_exact(pkv, name, filler):
    b = wl.make_workload(name, seed=0, filler=filler)
    g, _ = _gpu_step(pkv, b)
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    assert np.array_equal(host_bits(g["k_pool"]), k)
    assert np.array_equal(host_bits(g["v_pool"]), v)
    _status_ok(pkv)


@pytest.mark.parametrize("name,seed", [("tiny_decode", 0), ("tiny_decode", 1), ("tiny_decode", 2),
                                       ("cb_mix", 0), ("spec_verify", 0), ("sinks_scale", 0),
                                       ("cb_mix", 1), ("spec_verify", 2), ("prefill_mix", 0)])
def test_attention_matches_oracle(pkv, name, seed):
    b = wl.make_workload(name, seed=seed)
    _, out = _gpu_step(pkv, b)
    _, _, ref = _oracle_step(b)
    got = out.float().cpu().numpy()
    mx, mean = assert_close_to_oracle(got, ref, what=f"{name}/{seed}")
    print(f"{name} seed {seed}: max-abs {mx:.2e} mean-abs {mean:.2e}")
    _status_ok(pkv)


def test_ministral_layers_match_oracle(pkv):
    b = wl.make_workload("ministral_decode", seed=0, layers=4)
    for layer in range(b.layers):
        _, out = _gpu_step(pkv, b, layer)
        _, _, ref = _oracle_step(b, layer)
        assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"layer {layer}")
    _status_ok(pkv)


@pytest.mark.parametrize("name", ["tiny_decode", "sinks_scale"])
def test_float32_output(pkv, name):
    b = wl.make_workload(name, seed=3)
    _, out = _gpu_step(pkv, b, out_dtype=torch.float32)
    _, _, ref = _oracle_step(b)
    assert out.dtype == torch.float32
    assert_close_to_oracle(out.cpu().numpy(), ref, what=name)


@pytest.mark.parametrize("name", ["cb_mix", "spec_verify", "sinks_scale", "prefill_mix"])
def test_batch_vs_solo_bit_identical(pkv, name):
    b = wl.make_workload(name, seed=4)
    g, out = _gpu_step(pkv, b)
    full = host_bits(out)
    for s in range(b.num_seqs):
        sub = wl.select_seqs(b, [s])
        one = _attn_only(pkv, g, sub, tables=dev(sub.block_tables), lens=dev(sub.context_lens),
                         q=dev_bf16(sub.q[0]), q_starts=dev(sub.q_starts))
        r0, r1 = b.q_starts[s], b.q_starts[s + 1]
        assert np.array_equal(host_bits(one), full[r0:r1]), f"sequence {s} differs alone"
    _status_ok(pkv)


def test_window_rows_equal_single_row_decodes(pkv):
    b = wl.make_workload("spec_verify", seed=5)
    g, out = _gpu_step(pkv, b)
    full = host_bits(out)
    for s in range(0, b.num_seqs, 3):
        W, L = int(b.q_starts[s + 1] - b.q_starts[s]), int(b.context_lens[s])
        for w in range(W):
            r = int(b.q_starts[s]) + w
            one = pkv.paged_attention_forward(
                g["k_pool"], g["v_pool"], g["q"][r:r + 1].contiguous(), dev(np.array([0, 1], np.int32)),
                g["block_tables"][s:s + 1].contiguous(), dev(np.array([L - W + w + 1], np.int32)),
                max_context_len=L, max_q_rows_per_seq=1, causal=False)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(one)[0], full[r]), f"seq {s} row {w}"


def test_block_permutation_bit_identical(pkv):
    b = wl.make_workload("tiny_decode", seed=6)
    g, out = _gpu_step(pkv, b)
    k, v = host_bits(g["k_pool"]), host_bits(g["v_pool"])
    perm = np.random.default_rng(1).permutation(b.num_blocks)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    tables2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out2 = _attn_only(pkv, g, b, tables=dev(tables2), k_pool=dev_bf16(k2), v_pool=dev_bf16(v2))
    assert np.array_equal(host_bits(out2), host_bits(out))


def test_shared_prefix_vs_duplicated_blocks_bit_identical(pkv):
    b = wl.make_workload("cb_mix", seed=7)
    g, out = _gpu_step(pkv, b)
    k, v = host_bits(g["k_pool"]), host_bits(g["v_pool"])
    nsh = len(b.shared_block_ids)
    extra = nsh * len(b.sharing_seqs)
    k2 = np.concatenate([k, np.zeros((extra,) + k.shape[1:], np.uint16)])
    v2 = np.concatenate([v, np.zeros((extra,) + v.shape[1:], np.uint16)])
    tables2 = b.block_tables.copy()
    nxt = b.num_blocks
    for s in b.sharing_seqs:
        for j in range(nsh):
            k2[nxt], v2[nxt] = k[b.block_tables[s, j]], v[b.block_tables[s, j]]
            tables2[s, j] = nxt
            nxt += 1
    out2 = _attn_only(pkv, g, b, tables=dev(tables2), k_pool=dev_bf16(k2), v_pool=dev_bf16(v2))
    assert np.array_equal(host_bits(out2), host_bits(out))


@pytest.mark.parametrize("name", ["tiny_decode", "spec_verify", "sinks_scale"])
def test_nan_in_unused_slots_changes_nothing(pkv, name):
    a = wl.make_workload(name, seed=8, filler="random")
    n = wl.make_workload(name, seed=8, filler="nan")
    _, out_a = _gpu_step(pkv, a)
    _, out_n = _gpu_step(pkv, n)
    assert np.array_equal(host_bits(out_a), host_bits(out_n))


@pytest.mark.parametrize("d,bs", [(64, 16), (64, 32), (128, 16), (128, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths_all_variants(pkv, d, bs, causal):
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1024, 1025, 1537, 4097])
    W = np.array([1, 1, 3, 2, 16, 1, 5, 16, 1, 7, 2, 16, 4, 9]) if causal else np.ones(len(lens), np.int64)
    W = np.minimum(W, lens)
    b = wl.build_batch(11 + d + bs, name="ragged", lens=lens, n_new=W, q_rows=W, num_q_heads=16,
                       num_kv_heads=2, head_dim=d, block_size=bs, causal=causal, with_sinks=causal)
    _, out = _gpu_step(pkv, b)
    _, _, ref = _oracle_step(b)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"d{d} bs{bs} causal{causal}")
    _status_ok(pkv)


def test_contexts_beyond_sixty_four_splits(pkv):
    # 79, 137, 2 and 65 splits of 512 keys: the merge reloads (m, l) past 64 partials, and
    # both of its halves (odd and even split counts) are exercised
    lens = np.array([40001, 70000, 1000, 33000])
    W = np.array([1, 16, 1, 5])
    b = wl.build_batch(77, name="long", lens=lens, n_new=W, q_rows=W, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, block_size=16, causal=True, with_sinks=True)
    g, out = _gpu_step(pkv, b)
    _, _, ref = _oracle_step(b)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what="long contexts")
    full = host_bits(out)
    for s in (0, 1):
        sub = wl.select_seqs(b, [s])
        one = _attn_only(pkv, g, sub, tables=dev(sub.block_tables), lens=dev(sub.context_lens),
                         q=dev_bf16(sub.q[0]), q_starts=dev(sub.q_starts))
        assert np.array_equal(host_bits(one), full[b.q_starts[s]:b.q_starts[s + 1]]), f"sequence {s} alone"
    _status_ok(pkv)


def test_group_of_eight_with_sixteen_row_windows(pkv):
    lens = np.array([40, 700, 2049])
    W = np.array([16, 16, 9])
    b = wl.build_batch(21, name="m128", lens=lens, n_new=W, q_rows=W, num_q_heads=16, num_kv_heads=2,
                       head_dim=128, block_size=16, causal=True)
    _, out = _gpu_step(pkv, b)
    _, _, ref = _oracle_step(b)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what="G8xW16")


@pytest.mark.parametrize("d,bs", [(128, 16), (64, 32), (64, 16), (128, 32)])
def test_chunked_prefill_windows(pkv, d, bs):
    """Prefill chunks through the same kernel: W new rows appended, then attended causally
    (TensorSharp advanced features, section on chunked prefill: bounded chunks of 256)."""
    lens = np.array([256, 700, 1300, 3000])
    W = np.array([256, 200, 256, 97])
    b = wl.build_batch(41 + d, name="prefill", lens=lens, n_new=W, q_rows=W, num_q_heads=8, num_kv_heads=2,
                       head_dim=d, block_size=bs, causal=True)
    g, out = _gpu_step(pkv, b)
    _, _, ref = _oracle_step(b)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"prefill d{d}")
    # every prefill row equals its own one-row decode over the keys it may see
    full = host_bits(out)
    for s in (1, 3):
        for w in (0, 63, int(W[s]) - 1):
            r = int(b.q_starts[s]) + w
            one = pkv.paged_attention_forward(
                g["k_pool"], g["v_pool"], g["q"][r:r + 1].contiguous(), dev(np.array([0, 1], np.int32)),
                g["block_tables"][s:s + 1].contiguous(), dev(np.array([lens[s] - W[s] + w + 1], np.int32)),
                max_context_len=int(lens[s]), max_q_rows_per_seq=1)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(one)[0], full[r]), f"seq {s} row {w}"
    _status_ok(pkv)


def test_empty_context_and_sequences_without_rows(pkv):
    lens = np.array([0, 5, 9, 0])
    rows = np.array([1, 0, 2, 1])
    for sinks in (False, True):
        b = wl.build_batch(31, name="empty", lens=lens, n_new=np.zeros(4, np.int64), q_rows=rows,
                           num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16, causal=False,
                           with_sinks=sinks)
        _, out = _gpu_step(pkv, b)
        _, _, ref = _oracle_step(b)
        got = out.float().cpu().numpy()
        assert_close_to_oracle(got, ref, what=f"empty sinks={sinks}")
        assert np.all(got[0] == 0) and np.all(got[-1] == 0)
    _status_ok(pkv)


def test_explicit_head_map_and_scale(pkv):
    b = wl.make_workload("tiny_decode", seed=9)
    hmap = [1, 0, 1, 0, 0, 1, 1, 0]
    g, _ = _gpu_step(pkv, b)
    out = _attn_only(pkv, g, b, kv_head_of_q_head=hmap, scale=0.2)
    _, _, ref = _oracle_step(b, kv_head_of_q_head=np.array(hmap, np.int32), scale=0.2)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what="head map")


def test_workspace_is_reusable_across_calls(pkv):
    b = wl.make_workload("cb_mix", seed=10)
    g, out = _gpu_step(pkv, b)
    ws = pkv.new_attention_workspace(b.num_seqs, b.total_q_rows, b.num_q_heads, b.num_kv_heads,
                                     b.head_dim, b.max_context_len)
    outs = [host_bits(_attn_only(pkv, g, b, workspace=ws)) for _ in range(3)]
    assert all(np.array_equal(o, host_bits(out)) for o in outs)
    _status_ok(pkv)


def test_device_side_checks_report_and_do_not_fault(pkv):
    b = wl.make_workload("tiny_decode", seed=12)
    g, _ = _gpu_step(pkv, b)
    _status_ok(pkv)
    bad = b.block_tables.copy()
    bad[1, 0] = b.num_blocks + 5                         # block id outside the pool
    _attn_only(pkv, g, b, tables=dev(bad))
    rc, bits = pkv.device_status()
    assert rc == -5 and bits & 1
    lens = b.context_lens.copy()
    lens[2] = b.max_context_len + 40                     # longer than max_context_len
    _attn_only(pkv, g, b, lens=dev(lens))
    rc, bits = pkv.device_status()
    assert rc == -5 and bits & 2
    ws = pkv.new_attention_workspace(b.num_seqs, b.total_q_rows, b.num_q_heads, b.num_kv_heads,
                                     b.head_dim, b.max_context_len)
    ws.fill_(0x7f)                                       # leftover contents do not matter
    clean = host_bits(_attn_only(pkv, g, b))
    assert np.array_equal(host_bits(_attn_only(pkv, g, b, workspace=ws)), clean)
    _status_ok(pkv)
    qs = np.array([0, 1, 2, 3, 4], np.int32)
    qs2 = np.array([0, 2, 2, 3, 4], np.int32)            # 2 rows for sequence 0, max says 1
    _attn_only(pkv, g, b, q_starts=dev(qs2), max_rows=1)
    rc, bits = pkv.device_status()
    assert rc == -2 and bits & 4
    # the context is still healthy
    out = _attn_only(pkv, g, b, q_starts=dev(qs))
    _, _, ref = _oracle_step(b)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what="after checks")
    _status_ok(pkv)


def test_host_side_argument_errors(pkv):
    b = wl.make_workload("tiny_decode", seed=13)
    g = gpu_batch(b)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                    g["context_lens"], max_context_len=b.max_context_len,
                                    max_q_rows_per_seq=1, workspace=torch.zeros(256, dtype=torch.uint8,
                                                                                device="cuda"))
    assert e.value.status == -4
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                    g["context_lens"], max_context_len=10 ** 6, max_q_rows_per_seq=1)
    assert e.value.status == -2
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                    g["context_lens"], max_context_len=b.max_context_len,
                                    max_q_rows_per_seq=1, kv_head_of_q_head=[0] * 8)
    assert e.value.status == -2
    k96 = torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_forward(k96, k96, torch.zeros((1, 8, 96), dtype=torch.bfloat16, device="cuda"),
                                    g["q_starts"][:2].contiguous(), g["block_tables"][:1].contiguous(),
                                    g["context_lens"][:1].contiguous(), max_context_len=16,
                                    max_q_rows_per_seq=1)
    assert e.value.status == -3
