"""The C ABI without a GPU: the library builds, loads, exports what include/pkv.h declares,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import build, pkv as m
    build.build()
    m.lib()
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declarations_are_exported(pkv):
    names = _declared_functions()
    assert len(names) >= 9, names
    lib = pkv.lib()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"
    assert sorted(pkv.EXPORTED) == names
    assert lib.pkv_abi_version() == 2


def test_workspace_sizes(pkv):
    a = pkv.paged_attention_workspace_size(64, 64, 40, 8, 128, 32768)
    b = pkv.paged_attention_workspace_size(64, 64, 40, 8, 128, 65536)
    assert a % 256 == 0 and b > a > 64 * 40 * 64 * 128 * 4
    assert pkv.paged_attention_workspace_size(-1, 1, 1, 1, 64, 1) == 0
    assert pkv.spec_accept_workspace_size(136, 151936) % 256 == 0
    assert pkv.spec_accept_workspace_size(1, 0) == 0


def _pool(nb=4, bs=16, hkv=2, d=64, ptr=4096):
    return pkv_mod().__dict__["_Pool"](ptr, ptr, nb, bs, hkv, d)


def pkv_mod():
    from paged_kv_attention_forward_gb300 import pkv as m
    return m


def _attn(pkv, pool, **over):
    args = dict(q=4096, q_starts=4096, tables=4096, maxb=64, lens=4096, S=2, R=2, max_ctx=100,
                max_rows=1, Hq=8, hmap=None, sinks=None, causal=0, scale=0.0, out=4096, dt=0,
                ws=4096 * 64, ws_bytes=1 << 30)
    args.update(over)
    lib = pkv.lib()
    return lib.paged_attention_forward(
        ctypes.byref(pool), args["q"], args["q_starts"], args["tables"], args["maxb"], args["lens"],
        args["S"], args["R"], args["max_ctx"], args["max_rows"], args["Hq"], args["hmap"], args["sinks"],
        args["causal"], args["scale"], args["out"], args["dt"], args["ws"], args["ws_bytes"], None)


def test_host_validation_without_device(pkv):
    lib = pkv.lib()
    assert lib.paged_attention_forward(None, None, None, None, 0, None, 0, 0, 0, 0, 0, None, None, 0,
                                       0.0, None, 0, None, 0, None) == -1
    assert b"pool is NULL" in lib.pkv_last_error_string()
    assert _attn(pkv, _pool(d=96)) == -3
    assert _attn(pkv, _pool(bs=8)) == -3
    assert _attn(pkv, _pool(), Hq=7) == -2
    assert _attn(pkv, _pool(), dt=5) == -2
    assert _attn(pkv, _pool(), max_ctx=64 * 16 + 1) == -2
    assert _attn(pkv, _pool(), max_rows=1025, Hq=16) == -3          # G*rows = 8*1025 > 8192
    assert _attn(pkv, _pool(), q=None) == -1
    assert _attn(pkv, _pool(), out=4096 + 8) == -7
    assert _attn(pkv, _pool(), ws=4096 + 16) == -7
    assert _attn(pkv, _pool(), ws_bytes=100) == -4
    bad_map = (ctypes.c_int32 * 8)(0, 0, 0, 0, 0, 1, 1, 1)
    assert _attn(pkv, _pool(), hmap=ctypes.cast(bad_map, ctypes.c_void_p)) == -2
    assert b"exactly 4 q heads" in lib.pkv_last_error_string()
    assert _attn(pkv, _pool(), S=0) == 0                             # nothing to do
    p = _pool(d=7)
    assert lib.paged_kv_append(ctypes.byref(p), 4096, 4, 4096, 4096, 4096, 4096, 1, 1, None) == -3
    p = _pool()
    assert lib.paged_kv_append(ctypes.byref(p), 4096, 4, 4096, 4096, 4096 + 4, 4096, 1, 1, None) == -7
    assert lib.paged_kv_append(ctypes.byref(p), 4096, 4, 4096, 4096, 4096, 4096, 1, 0, None) == 0
    assert lib.spec_accept_greedy(4096, 0, 4096, 4096, 1, 1, 4096, 4096, 4096, 4096, 1 << 20, None) == -2
    assert lib.spec_accept_greedy(4096 + 4, 100, 4096, 4096, 1, 1, 4096, 4096, 4096, 4096, 1 << 20,
                                  None) == -7
    assert lib.spec_accept_greedy(4096, 100, 4096, 4096, 1, 1, 4096, 4096, 4096, 4096, 8, None) == -4
    # paged_block_hashes: argument checks that return before any CUDA call
    assert lib.paged_block_hashes(4096, None, 1, 16, 16, 0, None, 4096, 4, None) == -1
    assert lib.paged_block_hashes(4096, 4096, 1, 16, 0, 0, None, 4096, 4, None) == -3
    assert lib.paged_block_hashes(4096, 4096, 1, 16, 1025, 0, None, 4096, 4, None) == -3
    assert lib.paged_block_hashes(4096, 4096, -1, 16, 16, 0, None, 4096, 4, None) == -2
    assert lib.paged_block_hashes(4096, 4096, 1, 16, 16, 0, None, 4096 + 4, 4, None) == -7
    assert lib.paged_block_hashes(4096, 4096, 0, 16, 16, 0, None, 4096, 4, None) == 0
    # block allocation: checks made before any CUDA call
    bi = pkv._BlockIndexC(4096, 4096, 4096, 48, 4096, 4096)       # capacity not a power of two
    assert lib.paged_block_allocate(ctypes.byref(bi), 4096, 4096, 4096, 1, 16, 4, 4096, None, 4096, 1 << 20,
                                    None) == -2
    assert lib.paged_block_allocate(None, 4096, 4096, 4096, 1, 16, 4, 4096, None, 4096, 1 << 20, None) == -1
    bi.capacity = 64
    assert lib.paged_block_allocate(ctypes.byref(bi), 4096, 4096, 4096, 1, 16, 4, 4096, None, 4096, 8,
                                    None) == -4
    assert lib.paged_block_allocate(ctypes.byref(bi), 4096 + 4, 4096, 4096, 1, 16, 4, 4096, None, 4096, 1 << 20,
                                    None) == -7
    assert lib.paged_block_allocate(ctypes.byref(bi), 4096, 4096, 4096, 0, 16, 4, 4096, None, 4096, 1 << 20,
                                    None) == 0
    assert lib.paged_block_allocate_workspace_size(3, 5) == 256
    assert lib.paged_block_index_init(ctypes.byref(bi), -1, None) == -2
    # quantised pool: record size and the checks made before any CUDA call
    assert lib.pkv_qrecord_bytes(16, 128, 8) == 2 * 16 * 128 + 8 * 16
    assert lib.pkv_qrecord_bytes(32, 64, 4) == 2 * 32 * 32 + 8 * 32
    assert lib.pkv_qrecord_bytes(16, 64, 2) == 2 * 16 * 16 + 8 * 16
    assert lib.pkv_qrecord_bytes(16, 128, 2) == 2 * 16 * 32 + 8 * 16
    assert lib.pkv_qrecord_bytes(16, 128, 5) == 0
    qp = pkv._QPool(4096, 10, 16, 2, 128, 6)
    assert lib.paged_kv_append_quant(ctypes.byref(qp), 4096, 4, 4096, 4096, 4096, 4096, 1, 1, None) == -3
    qp.bits, qp.head_dim = 8, 96
    assert lib.paged_kv_append_quant(ctypes.byref(qp), 4096, 4, 4096, 4096, 4096, 4096, 1, 1, None) == -3
    qp.head_dim = 128
    assert lib.paged_kv_append_quant(ctypes.byref(qp), 4096, 4, 4096, 4096, 4096, 4096, 1, 0, None) == 0
    qp.records = 4096 + 8
    assert lib.paged_kv_append_quant(ctypes.byref(qp), 4096, 4, 4096, 4096, 4096, 4096, 1, 1, None) == -7
    assert lib.paged_attention_forward_quant(None, None, None, None, 0, None, 0, 0, 0, 0, 0, None, None, 0,
                                             0.0, None, 0, None, 0, None) == -1


def test_binding_refuses_host_tensors():
    # a host tensor must never reach the library as a device pointer
    import torch
    from paged_kv_attention_forward_gb300 import pkv
    k = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16)
    i32 = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        pkv.paged_kv_append(k, k, i32.view(2, 1), i32, torch.zeros(3, dtype=torch.int32), k[0], k[0])
    with pytest.raises(ValueError):
        pkv.paged_attention_forward(k, k, torch.zeros(1, 2, 64, dtype=torch.bfloat16), i32, i32.view(2, 1), i32,
                                    max_context_len=16, max_q_rows_per_seq=1)
    with pytest.raises(ValueError):
        pkv.paged_attention_forward_quant(torch.zeros(2, 1, pkv.qrecord_bytes(16, 64, 8), dtype=torch.uint8),
                                          16, 64, 8, torch.zeros(1, 2, 64, dtype=torch.bfloat16), i32,
                                          i32.view(2, 1), i32, max_context_len=16, max_q_rows_per_seq=1)
