"""Register budgets of the attention kernels, read from ptxas (-Xptxas -v).

The occupancy the design relies on for head_dim 128 holds only while these kernels stay
within their budgets without spills: 64-thread decode CTAs within 128 registers per thread
(eight CTAs per SM by registers; their 34 KB ring of two 32-key stages sets six), 128-thread
verify CTAs within 96 (five per SM), and the merge kernel (seven 128-thread CTAs per SM)
within 72.  A change that raises them slows every call without failing any numeric test.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_attention_forward_gb300", "csrc")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc")


def _ptxas_usage(src):
    out = subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                          "-I" + os.path.join(ROOT, "include"), "-Xptxas", "-v", "-c", src, "-o", os.devnull],
                         capture_output=True, text=True, cwd=CSRC, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    usage, cur = {}, None
    for line in out.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
        m = re.search(r"(\d+) bytes spill stores", line)
        if m and cur:
            usage.setdefault(cur, {})["spill"] = int(m.group(1))
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            usage.setdefault(cur, {})["regs"] = int(m.group(1))
    return usage


@pytest.fixture(scope="module")
def attention_usage():
    return _ptxas_usage("pkv_attention.cu")


def test_bf16_attention_kernels_fit_their_register_budget(attention_usage):
    usage = attention_usage
    # head_dim 128, block 16, bf16, no tree, no gather: the decode (1 row warp) and verify
    # (3 row warps) shapes of the cb_mix and spec_verify workloads
    pat = re.compile(r"paged_attention_kernelILi128ELi16ELi1ELi([13])ELi\d+ELb0ELi16ELi1ELb0E")
    found = {m.group(1): u for name, u in usage.items() for m in [pat.search(name)] if m}
    assert set(found) == {"1", "3"}, sorted(usage)[:5]
    budget = {"1": 128, "3": 96}
    for shape, u in found.items():
        assert u["regs"] <= budget[shape], f"{shape} row warps: {u['regs']} registers"
        assert u.get("spill", 0) == 0, f"{shape} row warps spill {u['spill']} bytes"


def test_merge_kernel_fits_its_register_budget(attention_usage):
    found = {name: u for name, u in attention_usage.items() if "paged_attention_combine_kernel" in name}
    assert len(found) == 2, sorted(attention_usage)[:5]   # head_dim 64 and 128
    for name, u in found.items():
        assert u["regs"] <= 72 and u.get("spill", 0) == 0, (name, u)
