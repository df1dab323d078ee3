"""Runs a synthetic case through the CUDA library (via the C ABI) and compares
with the oracle.  Test infrastructure: imports both sides, shares nothing
between them but the seeded inputs from ``synth``."""
from __future__ import annotations

import numpy as np

import synth

BF16_TOL = {"max_abs": 2e-2, "mean_abs": 2e-3}   # bf16 I/O, fp32 accumulation
FP8_TOL = {"max_abs": 6e-2, "mean_abs": 6e-3}    # fp8 KV cache
LSE_TOL = 2e-3                                   # fp32 log-sum-exp, absolute


def _torch():
    import torch
    return torch


def bf16_tensor(bits: np.ndarray, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def cache_tensor(arr: np.ndarray, device="cuda"):
    torch = _torch()
    if arr.dtype == np.uint16:
        return bf16_tensor(arr, device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_numpy_bits(t) -> np.ndarray:
    torch = _torch()
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(t) -> np.ndarray:
    return t.float().cpu().double().numpy()


def i32(a, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class GpuCase:
    """Device copy of a Case plus the library objects to run it."""

    def __init__(self, case: synth.Case, *, device="cuda", with_lse=True, num_sms=None):
        import paged_kv_variable_gb300 as pkv
        torch = _torch()
        self.case = case
        spec = case.spec
        self.pkv = pkv
        self.q = bf16_tensor(case.q, device)
        self.k_new = bf16_tensor(case.k_new, device) if case.k_new is not None else None
        self.v_new = bf16_tensor(case.v_new, device) if case.v_new is not None else None
        self.k_cache = cache_tensor(case.k_cache, device)
        self.v_cache = cache_tensor(case.v_cache, device)
        self.block_table = i32(case.block_table, device) if case.block_table is not None else None
        self.cu_q = i32(spec.cu_q, device)
        self.cu_new = i32(spec.cu_new, device)
        self.cache_lens = i32(spec.cache_lens, device)
        self.out = torch.full((spec.total_q, spec.hq, spec.d), float("nan"), dtype=torch.bfloat16, device=device)
        self.lse = (torch.full((spec.hq, max(1, spec.total_q)), float("nan"), dtype=torch.float32, device=device)
                    if with_lse else None)
        self.k_scale = torch.tensor([case.k_scale], dtype=torch.float32, device=device)
        self.v_scale = torch.tensor([case.v_scale], dtype=torch.float32, device=device)
        self.q_scale = (None if getattr(case, "q_scale", None) is None else
                        torch.tensor([case.q_scale], dtype=torch.float32, device=device))
        num_pages = case.num_pages if spec.paged else spec.batch
        self.problem = pkv.make_problem(batch=spec.batch, num_heads_q=spec.hq, num_heads_kv=spec.hkv,
                                        head_dim=spec.d, page_size=spec.page_size, cache_capacity=spec.capacity,
                                        num_pages=num_pages, cache_dtype=spec.cache_dtype, causal=spec.causal,
                                        softmax_scale=spec.softmax_scale)
        self.has_new = case.k_new is not None
        self.plan = pkv.plan(self.problem, spec.q_lens, spec.cache_lens, spec.new_lens if self.has_new else None,
                             num_sms)
        self.workspace = pkv.workspace_tensor(self.plan.workspace_bytes, device)
        self.plan.upload(self.workspace)

    def args(self, *, with_new=True):
        spec = self.case.spec
        return self.pkv.make_args(
            q=self.q, out=self.out, lse=self.lse, cu_seqlens_q=self.cu_q,
            max_seqlen_q=int(spec.q_lens.max()) if spec.batch else 0,
            k_cache=self.k_cache, v_cache=self.v_cache, cache_seqlens=self.cache_lens,
            k_new=self.k_new if with_new else None, v_new=self.v_new if with_new else None,
            cu_seqlens_knew=self.cu_new if with_new else None, block_table=self.block_table,
            k_scale=self.k_scale if spec.cache_dtype == "fp8" else None,
            v_scale=self.v_scale if spec.cache_dtype == "fp8" else None, q_scale=self.q_scale)

    def write_prefix(self):
        """fp8 cases: write the cached prefix with the library's own append."""
        case = self.case
        spec = case.spec
        if case.prefix_k is None or spec.cache_dtype != "fp8" or int(spec.cache_lens.sum()) == 0:
            return
        torch = _torch()
        zeros = torch.zeros(spec.batch, dtype=torch.int32, device=self.q.device)
        cu = i32(case.cu_prefix, self.q.device)
        a = self.pkv.make_args(q=None, out=None, cu_seqlens_q=None, max_seqlen_q=0, k_cache=self.k_cache,
                               v_cache=self.v_cache, cache_seqlens=zeros, k_new=bf16_tensor(case.prefix_k),
                               v_new=bf16_tensor(case.prefix_v), cu_seqlens_knew=cu, block_table=self.block_table,
                               k_scale=self.k_scale, v_scale=self.v_scale)
        self.pkv.kv_append(self.problem, a, int(spec.cache_lens.sum()), self.workspace)

    def run(self, stream=None):
        self.pkv.attn_varlen_kvcache_fwd(self.problem, self.args(), self.plan, self.workspace, stream=stream)

    def status(self) -> int:
        return self.pkv.get_status(self.workspace)


def compare_out(got_t, want: np.ndarray, tol: dict, what="out"):
    got = bf16_to_f64(got_t)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    max_abs = float(err.max()) if err.size else 0.0
    mean_abs = float(err.mean()) if err.size else 0.0
    assert max_abs <= tol["max_abs"], f"{what}: max-abs {max_abs:.3e} > {tol['max_abs']}"
    assert mean_abs <= tol["mean_abs"], f"{what}: mean-abs {mean_abs:.3e} > {tol['mean_abs']}"
    return max_abs, mean_abs


def compare_lse(got_t, want: np.ndarray, tol=LSE_TOL):
    got = got_t.cpu().double().numpy()[:, :want.shape[1]]
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), "lse: finite pattern differs"
    if fin.any():
        err = float(np.max(np.abs(got[fin] - want[fin])))
        assert err <= tol, f"lse max-abs {err:.3e} > {tol}"


def gpu_random_case(seed: int, *, cache_dtype="bf16", d=None, page_size=None, causal=None, max_cache=700,
                    max_new=80, sentinel="finite", with_new=True, q_equals_new=True, g=None, hkv=None):
    """Random case inside the library's supported set (D in {64,128}, either cache dtype; P drawn from 0, 16,
    32, 64, 256)."""
    rng = np.random.default_rng(seed)
    d = d or int(rng.choice([64, 128]))
    P = int(rng.choice([0, 16, 32, 64, 256])) if page_size is None else page_size
    hkv = hkv or int(rng.choice([1, 2, 4]))
    g = g or int(rng.choice([1, 2, 4, 8]))
    return synth.random_case(seed, batch=int(rng.integers(1, 6)), hq=hkv * g, hkv=hkv, d=d, page_size=P,
                             causal=causal, cache_dtype=cache_dtype, max_cache=max_cache, max_new=max_new,
                             with_new=with_new, sentinel=sentinel, q_equals_new=q_equals_new)
