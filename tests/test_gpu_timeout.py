"""The attention kernels' bounded-wait failure path, driven on the GPU without a fault.

Every wait inside the attention kernels has an iteration limit; when it runs out the kernel
records PKV_DEV_TIMEOUT, stops issuing copies, waits (with the default limit) for the copies
it already issued and returns, leaving the context usable.  pkv_debug_set_wait_limit(0)
makes every stage wait give up at once, so each call below takes that path on purpose: the
copies still land, only the waits give up.  The checks: the call reports PKV_ERR_TIMEOUT
with the timeout bit, and a normal call on the same context afterwards matches the float64
oracle.
"""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import assert_close_to_oracle, dev, dev_bf16, gpu_batch

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

PKV_ERR_TIMEOUT = -8
PKV_DEV_TIMEOUT = 16


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _attn(pkv, g, b):
    out = pkv.paged_attention_forward(
        g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"], g["context_lens"],
        max_context_len=b.max_context_len, max_q_rows_per_seq=b.max_q_rows_per_seq, sinks=g["sinks"],
        causal=b.causal)
    torch.cuda.synchronize()
    return out


def _expect_timeout_then_clean(pkv, run, ref):
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0, f"dirty status before the test: {rc}, {bits:#x}"
    pkv.debug_set_wait_limit(0)
    try:
        run()
        rc, bits = pkv.device_status()
    finally:
        pkv.debug_set_wait_limit(-1)
    assert rc == PKV_ERR_TIMEOUT and bits & PKV_DEV_TIMEOUT, (rc, bits)
    out = run()
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0, (rc, bits)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what="after the timeout")


@pytest.mark.parametrize("name,num_seqs", [("tiny_decode", None), ("spec_verify", 3)])
def test_bf16_waits_that_give_up_report_timeout(pkv, name, num_seqs):
    b = wl.make_workload(name, seed=31, num_seqs=num_seqs)
    g = gpu_batch(b)
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    ref = oracle.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens, sinks=b.sinks,
                                 causal=b.causal)
    _expect_timeout_then_clean(pkv, lambda: _attn(pkv, g, b), ref)


@pytest.mark.parametrize("bits,name,num_seqs", [(8, "tiny_decode", None), (4, "tiny_decode", None),
                                                (8, "spec_verify", 3), (4, "spec_verify", 3)])
def test_quantised_waits_that_give_up_report_timeout(pkv, bits, name, num_seqs):
    # Q8 records run two key-share consumer warps, Q4 three: their end-of-split merge
    # barriers are on the timeout path too; verify windows add the wide-row CTAs (Q8: two
    # row warps per key share, Q4: two n-tiles per row warp)
    b = wl.make_workload(name, seed=32, num_seqs=num_seqs)
    rec = wl.random_records(1, b, bits)[0]
    r = rec.copy()
    oracle.paged_kv_append_quant(r, b.block_size, b.head_dim, bits, b.block_tables, b.context_lens_old,
                                 b.new_starts, b.k_new[0], b.v_new[0])
    ref = oracle.paged_attention_quant(r, b.block_size, b.head_dim, bits, b.q[0], b.q_starts, b.block_tables,
                                       b.context_lens, sinks=b.sinks, causal=b.causal)
    g = dict(rec=dev(rec), tables=dev(b.block_tables), lens_old=dev(b.context_lens_old),
             lens=dev(b.context_lens), new_starts=dev(b.new_starts), q=dev_bf16(b.q[0]), q_starts=dev(b.q_starts))
    pkv.paged_kv_append_quant(g["rec"], b.block_size, b.head_dim, bits, g["tables"], g["lens_old"],
                              g["new_starts"], dev_bf16(b.k_new[0]), dev_bf16(b.v_new[0]))

    def run():
        out = pkv.paged_attention_forward_quant(
            g["rec"], b.block_size, b.head_dim, bits, g["q"], g["q_starts"], g["tables"], g["lens"],
            max_context_len=b.max_context_len, max_q_rows_per_seq=b.max_q_rows_per_seq)
        torch.cuda.synchronize()
        return out

    _expect_timeout_then_clean(pkv, run, ref)


def test_index_list_gather_waits_that_give_up_report_timeout(pkv):
    b = wl.make_workload("tiny_decode", seed=33)
    g = gpu_batch(b)
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    rng = np.random.default_rng(5)
    R = b.total_q_rows
    max_keys = 600
    counts = np.array([min(int(b.context_lens[s]), max_keys) for s in range(R)], np.int32)
    idx = np.zeros((R, max_keys), np.int32)
    for r in range(R):
        idx[r, :counts[r]] = np.sort(rng.choice(int(b.context_lens[r]), counts[r], replace=False))
    ref = oracle.paged_attention_sparse(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens, idx, counts)

    def run():
        out = pkv.paged_attention_forward_gather(g["k_pool"], g["v_pool"], g["q"], g["q_starts"],
                                                 g["block_tables"], g["context_lens"], dev(idx), dev(counts))
        torch.cuda.synchronize()
        return out

    _expect_timeout_then_clean(pkv, run, ref)
