"""Benchmark: one decode step of the continuous-batching mix through libpkv.so.

A step is the whole hot path on one batch: paged K/V append of every sequence's
new token, then paged attention of every decode row (and, for verify workloads,
the greedy accept).  Default workload: 64 sequences, cached lengths log-uniform
in [128, 32767] plus one appended token, 48 of them sharing a 2900-token prefix
through the same physical blocks, 40 q / 8 KV heads, head_dim 128, block 16.

Prints ONE JSON line (rank 0).  value = algorithmic bytes of the step / device
time of the step, in GB/s; algorithmic bytes count every distinct K/V token a
step must read once (shared prefix blocks once), plus q, out, the block-table
entries read, and the append's reads and writes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

--impl reference times the float64 CPU oracle (the checker) on the host cores on
a bounded sample of the same workload; it is a reported baseline, not a target.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
import types

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_attention_forward_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attention decode: achieved HBM GB/s (frac of GB300 peak), query-rows/s"
PROFILES = os.path.join(ROOT, "profiles")


# ---------------------------------------------------------------- accounting --
def kv_bytes_per_token_head(head_dim: int, bits: int) -> int:
    """K and V of one cached token of one KV head: bf16 rows, or its share of a
    quantised record (codes of K and V plus two float32 scales)."""
    return head_dim * 2 * 2 if bits == 16 else 2 * head_dim * bits // 8 + 8


def algorithmic_bytes(b: wl.PagedBatch, layers: int = 1, bits: int = 16) -> dict:
    """Bytes one step must move at least, per the workload's structure."""
    B, H, D = b.block_size, b.num_kv_heads, b.head_dim
    per_tok = kv_bytes_per_token_head(D, bits)
    shared = set(b.shared_block_ids.tolist())
    shared_tokens_read = 0
    if len(b.sharing_seqs):
        shared_tokens_read = len(shared) * B            # read once, not once per sharing sequence
    private_tokens = 0
    for s in range(b.num_seqs):
        L = int(b.context_lens[s])
        n_sh = len(shared) if s in set(b.sharing_seqs.tolist()) else 0
        private_tokens += L - n_sh * B
    kv = (private_tokens + shared_tokens_read) * H * per_tok
    logical_kv = int(b.context_lens.sum()) * H * per_tok
    list_bytes = 0
    if b.key_idx is not None:
        # index-list gather: every distinct physical (block, slot) the step's lists name, once
        row_seq = np.searchsorted(b.q_starts, np.arange(b.total_q_rows), side="right") - 1
        slots = set()
        for r in range(b.total_q_rows):
            s_ = row_seq[r]
            for t in b.key_idx[0, r, :b.key_counts[0, r]]:
                slots.add(int(b.block_tables[s_, t // B]) * B + int(t % B))
        kv = len(slots) * H * per_tok
        logical_kv = int(b.key_counts[0].sum()) * H * per_tok
        list_bytes = int(b.key_counts[0].sum()) * (4 + 4)    # the list entries and their table entries
    R = b.total_q_rows
    q_out = 2 * R * b.num_q_heads * D * 2
    table = int(sum((int(L) + B - 1) // B for L in b.context_lens)) * 4 + (b.num_seqs * 2 + 1) * 4
    if b.key_idx is not None:
        table = list_bytes + (b.num_seqs * 2 + 1) * 4 + b.total_q_rows * 4
    r_new = int(b.new_starts[-1])
    append = r_new * H * (D * 2 * 2 + per_tok)          # read k_new/v_new, write the pool slots
    attn = kv + q_out + table
    accept = 0
    if b.logits is not None:
        accept = b.logits.size * 4 + R * 4 * (3 if b.parents is None else 5)
    return dict(attention=attn * layers, append=append * layers, accept=accept,
                step=(attn + append) * layers + accept, kv_unique=kv * layers,
                kv_logical=logical_kv * layers, rows=R)


def algorithmic_flops(b: wl.PagedBatch) -> float:
    """Floating-point operations of one attention call: for every (row, q head), q·k and
    p·v over each key the row sees, 4·d per key (the softmax's own work not counted)."""
    keys = 0
    for s in range(b.num_seqs):
        r0, r1 = int(b.q_starts[s]), int(b.q_starts[s + 1])
        W, L = r1 - r0, int(b.context_lens[s])
        for w in range(W):
            r = r0 + w
            if b.key_idx is not None:
                n = int(b.key_counts[0, r])
            elif b.tree_masks is not None:
                n = L - W + bin(int(b.tree_masks[r]) & ((1 << W) - 1)).count("1")
            elif b.causal:
                n = L - W + w + 1
            else:
                n = L
            keys += n
    return 4.0 * b.head_dim * b.num_q_heads * keys


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return {}


def stored_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it matches the current sources."""
    from paged_kv_attention_forward_gb300 import build
    path = os.path.join(PROFILES, f"{kernel}_{workload}.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    vals = {}
    for ln in lines:
        if ":" in ln and not ln.startswith("#"):
            k, _, v = ln.partition(":")
            vals[k.strip()] = v.strip()
    if vals.get("source_digest") != build.source_digest(build.ATTENTION_SOURCES):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- multi-rank --
def replica_seed(seed: int, rank: int) -> int:
    """Each rank runs its own replica of the workload (weak scaling): same shape, own data."""
    return seed + rank


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (the job is as slow as its slowest rank)."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, each rank processing units_per_rank per step."""
    return world * units_per_rank / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ our arm --
def run_ours(args, rank, world, local_rank):
    import torch
    from paged_kv_attention_forward_gb300 import pkv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if getattr(args, "kernel", "mma") == "tcgen05":
        pkv.set_attention_kernel(pkv.PKV_KERNEL_TCGEN05)
    layers = 40 if args.workload == "ministral_decode" else 1
    b = wl.make_workload(args.workload, seed=replica_seed(args.seed, rank), layers=layers,
                         num_seqs=args.num_seqs)
    bits = args.kv_bits
    quant = bits != 16
    acct = algorithmic_bytes(b, layers, bits)

    def d_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    if quant:
        recs = wl.random_records(replica_seed(args.seed, rank) + 7, b, bits, layers)
        records = [d(recs[i]) for i in range(layers)]
        del recs
    else:
        pools = [(d_bf16(b.k_pool[i]), d_bf16(b.v_pool[i])) for i in range(layers)]
    tables, lens_old, lens = d(b.block_tables), d(b.context_lens_old), d(b.context_lens)
    new_starts, q_starts = d(b.new_starts), d(b.q_starts)
    k_new = [d_bf16(b.k_new[i]) for i in range(layers)]
    v_new = [d_bf16(b.v_new[i]) for i in range(layers)]
    qs = [d_bf16(b.q[i]) for i in range(layers)]
    sinks = None if b.sinks is None else d(b.sinks)
    outs = [torch.empty_like(q) for q in qs]
    ws = pkv.new_attention_workspace(b.num_seqs, b.total_q_rows, b.num_q_heads, b.num_kv_heads,
                                     b.head_dim, b.max_context_len if b.key_idx is None else b.key_idx.shape[2], dev)
    logits = drafts = acc_ws = None
    acc_out = None
    tree = b.tree_masks is not None
    tree_masks = d(b.tree_masks.view(np.int32)) if tree else None
    parents = d(b.parents) if tree else None
    positions = None
    if b.logits is not None:
        logits, drafts = d(b.logits), d(b.draft_tokens)
        acc_ws = torch.empty(pkv.sampled_accept_workspace_size(b.total_q_rows, b.logits.shape[1]),
                             dtype=torch.uint8, device=dev)
        # absolute position of the token each verify row draws: L - W + w + 1
        row_seq = np.searchsorted(b.q_starts, np.arange(b.total_q_rows), side="right") - 1
        w_of = np.arange(b.total_q_rows) - b.q_starts[row_seq]
        positions = d((b.context_lens[row_seq] - np.diff(b.q_starts)[row_seq] + w_of + 1).astype(np.int32))
        acc_out = tuple(torch.empty(n, dtype=torch.int32, device=dev)
                        for n in (b.total_q_rows, b.num_seqs, b.total_q_rows, b.total_q_rows))
    has_append = int(b.new_starts[-1]) > 0
    gather = b.key_idx is not None
    if gather:
        key_sets = [d(b.key_idx[k]) for k in range(b.key_idx.shape[0])]
        key_counts = d(b.key_counts[0])
        step_no = [0]
    accept_mode = getattr(args, "accept", "greedy")
    max_ctx, max_rows = b.max_context_len, b.max_q_rows_per_seq
    stream = torch.cuda.current_stream()
    # per layer: append (if any) + attention split kernel + attention merge kernel; accept: 2
    accept_launches = {"greedy": 2, "sampled": 3, "sampled-topkp": 4}[accept_mode] if logits is not None else 0
    launches_per_step = layers * (int(has_append) + 2) + accept_launches

    # the tensors a step reads and writes: one set for the device-timed region; the end-to-end
    # pass alternates two sets so that one step's copies overlap the other's compute
    io = types.SimpleNamespace(tables=tables, lens_old=lens_old, lens=lens, new_starts=new_starts,
                               q_starts=q_starts, k_new=k_new, v_new=v_new, qs=qs, outs=outs, logits=logits,
                               drafts=drafts, acc_out=acc_out, tree_masks=tree_masks, parents=parents,
                               positions=positions, keys=None)

    def step(ev_pairs=None, li=None, io=io, st=None, attn_only=False):
        st = stream if st is None else st
        for i in range(layers):
            if attn_only:
                pass
            elif has_append and quant:
                pkv.paged_kv_append_quant(records[i], b.block_size, b.head_dim, bits, io.tables, io.lens_old,
                                          io.new_starts, io.k_new[i], io.v_new[i], stream=st)
            elif has_append:
                pkv.paged_kv_append(pools[i][0], pools[i][1], io.tables, io.lens_old, io.new_starts, io.k_new[i],
                                    io.v_new[i], stream=st)
            if ev_pairs is not None:
                ev_pairs[li][0].record(st)
            if gather:
                k_set = io.keys
                if k_set is None:   # device-timed region: the lists change every step
                    k_set = key_sets[step_no[0] % len(key_sets)]
                    step_no[0] += 1
                pkv.paged_attention_forward_gather(pools[i][0], pools[i][1], io.qs[i], io.q_starts, io.tables,
                                                   io.lens, k_set, key_counts, sinks=sinks, out=io.outs[i],
                                                   workspace=ws, stream=st)
            elif quant:
                pkv.paged_attention_forward_quant(records[i], b.block_size, b.head_dim, bits, io.qs[i], io.q_starts,
                                                  io.tables, io.lens, max_context_len=max_ctx,
                                                  max_q_rows_per_seq=max_rows, sinks=sinks, causal=b.causal,
                                                  out=io.outs[i], workspace=ws, stream=st)
            elif tree:
                pkv.paged_tree_attention_forward(pools[i][0], pools[i][1], io.qs[i], io.q_starts, io.tables, io.lens,
                                                 io.tree_masks, max_context_len=max_ctx,
                                                 max_q_rows_per_seq=max_rows, sinks=sinks, out=io.outs[i],
                                                 workspace=ws, stream=st)
            else:
                pkv.paged_attention_forward(pools[i][0], pools[i][1], io.qs[i], io.q_starts, io.tables, io.lens,
                                            max_context_len=max_ctx, max_q_rows_per_seq=max_rows, sinks=sinks,
                                            causal=b.causal, out=io.outs[i], workspace=ws, stream=st)
            if ev_pairs is not None:
                ev_pairs[li][1].record(st)
                li += 1
        if attn_only:
            return li
        if io.logits is not None and accept_mode in ("sampled", "sampled-topkp"):
            filt = dict(top_k=50, top_p=0.9) if accept_mode == "sampled-topkp" else {}
            pkv.spec_accept_sampled(io.logits, io.q_starts, io.drafts, io.positions, seed=args.seed + 1,
                                    temperature=1.0, min_p=0.05, **filt, parents=io.parents,
                                    sampled_out=io.acc_out[0], accept_len=io.acc_out[1], out_tokens=io.acc_out[2],
                                    accepted_rows=io.acc_out[3], workspace=acc_ws, stream=st)
        elif io.logits is not None and tree:
            pkv.spec_accept_tree_greedy(io.logits, io.q_starts, io.drafts, io.parents, argmax_out=io.acc_out[0],
                                        accept_len=io.acc_out[1], out_tokens=io.acc_out[2],
                                        accepted_rows=io.acc_out[3], workspace=acc_ws, stream=st)
        elif io.logits is not None:
            pkv.spec_accept_greedy(io.logits, io.q_starts, io.drafts, argmax_out=io.acc_out[0],
                                   accept_len=io.acc_out[1], out_tokens=io.acc_out[2], workspace=acc_ws, stream=st)
        return li

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    rc, dev_bits = pkv.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {dev_bits:#x} after warm-up")

    # ---- device-resident timed region ----
    # By default the step is captured as a CUDA graph and replayed, as a serving loop replays
    # its decode step (its launches then cost one graph launch).  The per-call durations for
    # the roofline come from a graph of the step's attention calls alone (no appends, no
    # accept), several passes over the layers back to back, timed by CUDA events around its
    # replays: the calls' own GPU time, without the host's launch gaps that an eager call of a
    # few microseconds also measures (an eager pass, one event pair per call, is reported
    # beside it).  The index-list gather, whose lists change every step, captures one graph
    # per list set and replays them in turn.  --eager: plain launches throughout, and the
    # per-call times come from the timed region's own event pairs.
    graph = not getattr(args, "eager", False)

    def capture(io_, fn=None):
        fn = fn or (lambda st_: step(io=io_, st=st_))
        g_ = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn(side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g_):
            fn(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g_

    n_eager = min(args.steps, 200) if graph else args.steps
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_eager * layers)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        li = 0
        for _ in range(n_eager):
            li = step(ev_pairs, li)
        torch.cuda.synchronize()
        if gather:
            g_steps = [capture(types.SimpleNamespace(**{**vars(io), "keys": ks})) for ks in key_sets]
        else:
            g_steps = [capture(io)]
        for k in range(3):
            g_steps[k % len(g_steps)].replay()
        # the attention calls alone, back to back (about 200 calls per replay)
        io_attn = types.SimpleNamespace(**{**vars(io), "keys": key_sets[0]}) if gather else io
        reps = max(1, 200 // layers)

        def attn_passes(st_):
            for _ in range(reps):
                step(io=io_attn, st=st_, attn_only=True)

        g_attn = capture(io_attn, attn_passes)
        g_attn.replay()
        n_attn_replays = 3
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_attn_replays):
            g_attn.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        attn_graph_calls = n_attn_replays * reps * layers
        attn_graph_ms = a0.elapsed_time(a1) / attn_graph_calls
        del g_attn
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    t0.record(stream)
    li = 0
    for i in range(args.steps):
        if graph:
            g_steps[i % len(g_steps)].replay()
        else:
            li = step(ev_pairs, li)
    t1.record(stream)
    barrier()
    wall1 = time.perf_counter()
    clock_info = clocks.stop() if clocks else None
    ms_total = t0.elapsed_time(t1)
    attn_ms = [a.elapsed_time(z) for a, z in ev_pairs]
    rc, dev_bits = pkv.device_status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {dev_bits:#x} after timed steps")

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory and its results back.  Two sets of
    # device buffers let step i + 1's input copies (on a copy stream) overlap step i's kernels,
    # and step i's result copies overlap step i + 1's kernels, as a serving loop would.
    # Each set's inputs live in one packed device buffer (and its results in another), so
    # a step moves its inputs with one host-to-device copy and its results with one copy back.
    in_items = [("tables", b.block_tables), ("lens_old", b.context_lens_old), ("lens", b.context_lens),
                ("new_starts", b.new_starts), ("q_starts", b.q_starts)]
    in_items += [(("qs", li), np.ascontiguousarray(b.q[li]).view(np.int16)) for li in range(layers)]
    in_items += [(("k_new", li), np.ascontiguousarray(b.k_new[li]).view(np.int16)) for li in range(layers)]
    in_items += [(("v_new", li), np.ascontiguousarray(b.v_new[li]).view(np.int16)) for li in range(layers)]
    if logits is not None:
        in_items += [("logits", b.logits), ("drafts", b.draft_tokens), ("positions", positions.cpu().numpy())]
    if tree:
        in_items += [("tree_masks", b.tree_masks.view(np.int32)), ("parents", b.parents)]
    if gather:   # this step's lists come from the host too
        in_items.append(("keys", b.key_idx[0]))
    out_items = [(("outs", li), (b.total_q_rows, b.num_q_heads, b.head_dim), np.int16) for li in range(layers)]
    if acc_out is not None:
        out_items += [(("acc_out", n), tuple(t.shape), np.int32) for n, t in enumerate(acc_out)]

    def layout(sizes):
        offs, at = [], 0
        for nbytes in sizes:
            offs.append(at)
            at += (nbytes + 255) // 256 * 256
        return offs, at

    in_offs, in_total = layout([np.asarray(a).nbytes for _, a in in_items])
    out_offs, out_total = layout([int(np.prod(shape)) * np.dtype(dt).itemsize for _, shape, dt in out_items])
    h_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    h_in_np = h_in.numpy()
    for (_, a), off in zip(in_items, in_offs):
        raw = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        h_in_np[off:off + raw.size] = raw
    h_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_in = [torch.empty(in_total, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(out_total, dtype=torch.uint8, device=dev) for _ in range(2)]
    to_torch = {np.dtype(np.int32): torch.int32, np.dtype(np.int16): torch.int16}

    def view(buf, off, a_dtype, shape, bf16=False):
        n = int(np.prod(shape)) * np.dtype(a_dtype).itemsize
        t = buf[off:off + n].view(to_torch[np.dtype(a_dtype)]).view(shape)
        return t.view(torch.bfloat16) if bf16 else t

    def make_set(k):
        st_ = types.SimpleNamespace(qs=[None] * layers, k_new=[None] * layers, v_new=[None] * layers,
                                    outs=[None] * layers, acc_out=None if acc_out is None else [None] * len(acc_out),
                                    logits=None, drafts=None, positions=None, tree_masks=None, parents=None,
                                    keys=None)
        for (name, a), off in zip(in_items, in_offs):
            a = np.asarray(a)
            if isinstance(name, tuple):
                getattr(st_, name[0])[name[1]] = view(d_in[k], off, np.int16, a.shape, bf16=True)
            elif name == "logits":
                st_.logits = d_in[k][off:off + a.nbytes].view(torch.float32).view(a.shape)
            else:
                setattr(st_, name, view(d_in[k], off, np.int32, a.shape))
        for (name, shape, dt), off in zip(out_items, out_offs):
            getattr(st_, name[0])[name[1]] = view(d_out[k], off, dt, shape, bf16=name[0] == "outs")
        if st_.acc_out is not None:
            st_.acc_out = tuple(st_.acc_out)
        return st_

    sets = [make_set(0), make_set(1)]
    g_sets = [capture(sets[0]), capture(sets[1])] if graph else None
    h2d = in_total
    d2h = out_total
    copy_stream = torch.cuda.Stream()

    def copy_in(k):
        d_in[k].copy_(h_in, non_blocking=True)

    def copy_out(k):
        h_out[k].copy_(d_out[k], non_blocking=True)

    def e2e_run(n):
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_stream.wait_stream(stream)
        e0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            copy_in(0)
        ready[0].record(copy_stream)
        for i in range(n):
            k, o = i % 2, 1 - i % 2
            stream.wait_event(ready[k])
            if graph:
                g_sets[k].replay()
            else:
                step(io=sets[k])
            done[k].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(done[o])   # step i - 1 has finished with set o
                    copy_in(o)
                    ready[o].record(copy_stream)
                copy_stream.wait_event(done[k])
                copy_out(k)
        e1.record(copy_stream)
        return e0, e1

    e2e_steps = max(2, min(args.steps, args.e2e_steps))
    e2e_run(max(3, args.warmup // 4))
    barrier()
    e0, e1 = e2e_run(e2e_steps)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)

    # ---- max over ranks ----
    ms_per_step = ms_total / args.steps
    e2e_ms_per_step = e2e_ms / e2e_steps
    attn_eager_ms = statistics.fmean(attn_ms)
    attn_avg_ms = attn_graph_ms if graph else attn_eager_ms
    ms_per_step, e2e_ms_per_step, attn_avg_ms, attn_eager_ms = max_over_ranks(
        [ms_per_step, e2e_ms_per_step, attn_avg_ms, attn_eager_ms], dist, dev)
    if rank != 0:
        return None

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_kind = "measured"
    if peak is None:
        peak, peak_kind = 6800.0, "fallback"
    per_launch_bytes = acct["attention"] / layers
    achieved = per_launch_bytes / (attn_avg_ms * 1e-3) / 1e9
    flops = algorithmic_flops(b)
    attn_tflops = flops / (attn_avg_ms * 1e-3) / 1e12
    kernel_tag = ("paged_attention" if not quant else f"paged_attention_q{bits}") + (
        "_tcgen05" if getattr(args, "kernel", "mma") == "tcgen05" and not quant else "")
    traffic = stored_traffic(kernel_tag, args.workload)
    value = whole_job_rate(acct["step"], world, ms_per_step) / 1e9
    e2e_value = whole_job_rate(acct["step"], world, e2e_ms_per_step) / 1e9
    rows_per_s = whole_job_rate(acct["rows"] * layers, world, ms_per_step)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_description(b, layers)
                   + ("" if not gather else f", index-list gather: [last 128 | 512 older] keys per row, "
                                            f"{b.key_idx.shape[0]} list sets used in turn"),
                   "global_batch": b.num_seqs * world,
                   "seq_len": b.max_context_len, "parallelism": f"dp{world} (independent replicas)",
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB); no flush",
                   "seed": args.seed,
                   "accept": None if b.logits is None else accept_mode,
                   "launch": "cuda graph (one captured step, replayed)" if graph else "eager",
                   "kv_codec": "bf16" if not quant else f"q{bits} (per-row float32 scale)",
                   "kernel": "tcgen05" if getattr(args, "kernel", "mma") == "tcgen05" and not quant else "mma.sync"},
        "query_rows_per_s": round(rows_per_s, 1),
        "frac_of_measured_hbm": round(value / peak, 4),
        "frac_of_nominal_8tbs": round(value / 8000.0, 4),
        "bytes_per_step": acct["step"], "kv_unique_bytes_per_step": acct["kv_unique"],
        "kv_logical_bytes_per_step": acct["kv_logical"],
        "attention_tflops": round(attn_tflops, 2), "flops_per_launch": flops,
        "roofline": {"kernel": "paged attention call (split kernel + merge kernel)"
                     + ("" if not quant else f", q{bits} records"), "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} (hbm_gbs, copy kernel)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "bytes_per_launch": per_launch_bytes,
                     "avg_launch_ms": round(attn_avg_ms, 5),
                     "launches_timed": attn_graph_calls if graph else len(attn_ms),
                     "launches_timed_mode": ("a graph of the step's attention calls alone, replayed back to back "
                                             "before the timed steps" if graph else "timed region"),
                     "avg_launch_ms_eager": round(attn_eager_ms, 5),
                     "traffic": traffic},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms_per_step, 5),
                "steps": e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_info,
        "wall_s_timed_region": round(wall1 - wall0, 3),
    }
    # a call whose flops per byte exceed the ridge of the measured peaks (prefill chunks) is a
    # dense contraction: its roofline is the tensor pipe's
    tpeak = peaks.get("bf16_tflops")
    tkind = "measured (bf16_tflops, cuBLAS bf16 GEMM, burst)"
    if tpeak is None:
        tpeak, tkind = 1900.0, "fallback"
    if flops / per_launch_bytes > tpeak * 1e12 / (peak * 1e9):
        line["roofline"].update(bound="tensor", achieved=round(attn_tflops, 2), peak=tpeak, peak_kind=tkind,
                                unit="TFLOP/s", frac=round(attn_tflops / tpeak, 4),
                                hbm_achieved_gbs=round(achieved, 2))
    return line


def workload_description(b, layers):
    return (f"{b.name}: {b.num_seqs} seqs, context {int(b.context_lens.min())}-{int(b.context_lens.max())} "
            f"(sum {int(b.context_lens.sum())}), {b.num_q_heads} q / {b.num_kv_heads} kv heads, "
            f"head_dim {b.head_dim}, block {b.block_size}, rows {b.total_q_rows}, "
            f"appended {int(b.new_starts[-1])}, shared prefix blocks {len(b.shared_block_ids)} "
            f"x {len(b.sharing_seqs)} seqs, layers {layers}, causal {int(b.causal)}, "
            f"sinks {int(b.sinks is not None)}")


# ------------------------------------------------------------ oracle timing --
def time_oracle_step(sub: wl.PagedBatch, threads: int, records=None, bits: int = 16):
    import oracle
    # the append writes the same values into the same slots on every call, so the pool is
    # used in place (copying a whole pool per step would cost more than the step)
    if records is not None:
        rec = records
        t = time.perf_counter()
        if int(sub.new_starts[-1]) > 0:
            oracle.paged_kv_append_quant(rec, sub.block_size, sub.head_dim, bits, sub.block_tables,
                                         sub.context_lens_old, sub.new_starts, sub.k_new[0], sub.v_new[0])
        oracle.paged_attention_quant(rec, sub.block_size, sub.head_dim, bits, sub.q[0], sub.q_starts,
                                     sub.block_tables, sub.context_lens, sinks=sub.sinks, causal=sub.causal,
                                     num_threads=threads)
        return time.perf_counter() - t
    k, v = sub.k_pool[0], sub.v_pool[0]
    t = time.perf_counter()
    if int(sub.new_starts[-1]) > 0:
        oracle.paged_kv_append(k, v, sub.block_tables, sub.context_lens_old, sub.new_starts,
                               sub.k_new[0], sub.v_new[0])
    if sub.key_idx is not None:
        oracle.paged_attention_sparse(k, v, sub.q[0], sub.q_starts, sub.block_tables, sub.context_lens,
                                      sub.key_idx[0], sub.key_counts[0], sinks=sub.sinks)
    else:
        oracle.paged_attention(k, v, sub.q[0], sub.q_starts, sub.block_tables, sub.context_lens, sinks=sub.sinks,
                               causal=sub.causal, num_threads=threads, tree_masks=sub.tree_masks)
    if sub.logits is not None and sub.parents is not None:
        oracle.spec_accept_tree_greedy(sub.logits, sub.q_starts, sub.draft_tokens, sub.parents)
    elif sub.logits is not None:
        oracle.spec_accept_greedy(sub.logits, sub.q_starts, sub.draft_tokens)
    return time.perf_counter() - t


def cpu_baseline(b: wl.PagedBatch, budget_s: float = 12.0, max_runs: int = 60, bits: int = 16, seed: int = 0):
    """The oracle, as it stands, on the whole batch, repeated for about budget_s seconds."""
    import oracle
    oracle.build_oracle()
    threads = len(os.sched_getaffinity(0))
    acct = algorithmic_bytes(b, 1, bits)
    records = wl.random_records(seed + 7, b, bits)[0] if bits != 16 else None
    times = []
    t_start = time.perf_counter()
    while len(times) < max_runs and (not times or time.perf_counter() - t_start < budget_s):
        times.append(time_oracle_step(b, threads, records, bits))
    med = statistics.median(times)
    return {"value": round(acct["step"] / med / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"the whole batch ({b.num_seqs} seqs, {int(b.context_lens.sum())} cached tokens): "
                       f"append + attention{' + accept' if b.logits is not None else ''} in float64, "
                       f"median of {len(times)} runs ({med:.2f} s each, {sum(times):.1f} s in all)")}


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores, rank 0 only."""
    if rank != 0:
        return None
    import oracle
    oracle.build_oracle()
    layers = 1
    b = wl.make_workload(args.workload, seed=args.seed, layers=layers, num_seqs=args.num_seqs)
    threads = len(os.sched_getaffinity(0))
    # size the per-step sample so that warm-up + timed steps take about 90 s in all
    order = np.random.default_rng(12345).permutation(b.num_seqs)
    cal = wl.select_seqs(b, order[:1])
    t_cal = max(time_oracle_step(cal, threads), 1e-4)
    tok_per_s = int(cal.context_lens.sum()) / t_cal
    budget_tokens = tok_per_s * 90.0 / (args.steps + args.warmup)
    chosen, tokens = [], 0
    for s in order:
        if tokens + int(b.context_lens[s]) > budget_tokens:
            continue
        chosen.append(int(s))
        tokens += int(b.context_lens[s])
    if not chosen:   # nothing fits: the shortest sequence alone
        chosen = [int(np.argmin(b.context_lens))]
    sub = wl.select_seqs(b, sorted(chosen))
    acct = algorithmic_bytes(sub)
    for _ in range(args.warmup):
        time_oracle_step(sub, threads)
    times = [time_oracle_step(sub, threads) for _ in range(args.steps)]
    total = sum(times)
    value = acct["step"] * args.steps / total / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_description(b, layers), "global_batch": b.num_seqs,
                   "seq_len": b.max_context_len, "parallelism": "host cores", "seed": args.seed},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{sub.num_seqs} of the batch's sequences ({int(sub.context_lens.sum())} "
                                   f"cached tokens) per step, chosen in a fixed random order to fit "
                                   f"about 90 s for all steps; append + attention in float64"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=wl.WORKLOADS, default="cb_mix")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="resize the batch (same per-sequence distribution); for profiling smaller cases")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=("mma", "tcgen05"), default="mma",
                    help="kernel of the bf16 attention calls (pkv_set_attention_kernel)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every kernel of every step directly instead of replaying a captured CUDA graph")
    ap.add_argument("--kv-bits", type=int, choices=(16, 8, 4, 2), default=16,
                    help="16: bf16 K/V pools; 8 / 4 / 2: quantised KV blocks (Q8 / Q4 / Q2 records)")
    ap.add_argument("--accept", choices=("greedy", "sampled", "sampled-topkp"), default="greedy",
                    help="verify workloads: greedy accept, keyed sampling at T = 1, min_p = 0.05, or the same "
                         "with top_k = 50 and top_p = 0.9")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        if not args.no_cpu_baseline and world == 1:
            b = wl.make_workload(args.workload, seed=args.seed, layers=1, num_seqs=args.num_seqs)
            line["cpu_baseline"] = cpu_baseline(b, bits=args.kv_bits, seed=args.seed)
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
