"""Shared test helpers: moving generator output to the GPU and comparing with the oracle."""
import numpy as np

TOL_MAX = 2e-2   # max-abs error of bf16 attention output vs the float64 oracle
TOL_MEAN = 2e-3  # mean-abs error


def dev_bf16(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t):
    """bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_batch(b, layer=0, device="cuda"):
    """Device copies of one layer of a PagedBatch."""
    return dict(
        k_pool=dev_bf16(b.k_pool[layer], device), v_pool=dev_bf16(b.v_pool[layer], device),
        block_tables=dev(b.block_tables, device), context_lens_old=dev(b.context_lens_old, device),
        context_lens=dev(b.context_lens, device), new_starts=dev(b.new_starts, device),
        k_new=dev_bf16(b.k_new[layer], device), v_new=dev_bf16(b.v_new[layer], device),
        q_starts=dev(b.q_starts, device), q=dev_bf16(b.q[layer], device),
        sinks=None if b.sinks is None else dev(b.sinks, device))


def assert_close_to_oracle(got, ref, tol_max=TOL_MAX, tol_mean=TOL_MEAN, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= tol_max, f"{what}: max-abs error {err.max():.3e} > {tol_max}"
    assert err.mean() <= tol_mean, f"{what}: mean-abs error {err.mean():.3e} > {tol_mean}"
    return float(err.max()), float(err.mean())
