"""Shared helpers for the parity tests: move seeded workloads to the GPU, run
the oracle on the same inputs, and compare with the stated tolerances.

Tolerances (attention outputs, bf16 inputs, fp64 oracle): max abs error
<= 1e-2 and relative L2 error <= 5e-3 per row, a row being one (token, query
head) vector of head_dim values.  Integer and byte results are bit-exact."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import paged_attention as pa
from oracle import sampler as sm

ATOL_MAX = 1e-2
REL_L2_ROW = 5e-3
# Sampler ids: exact on every row whose oracle log-margin between the two best
# candidates exceeds NEAR_TIE (far above fp32 rounding of the kernel's key);
# on a near-tie row either of the two best is accepted, and such rows are counted.
NEAR_TIE = 1e-4


def f32(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor -> float32 numpy (exact for bf16)."""
    return t.detach().to("cpu").float().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns, so NaN payloads compare too."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def assert_attention_close(out: torch.Tensor, ref: np.ndarray, what: str = ""):
    got = out.detach().to("cpu").double().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    d = got.shape[-1]
    g2 = got.reshape(-1, d)
    r2 = ref.reshape(-1, d)
    num = np.linalg.norm(g2 - r2, axis=1)
    den = np.maximum(np.linalg.norm(r2, axis=1), 1e-30)
    rel = num / den
    worst = float(rel.max()) if rel.size else 0.0
    assert max_abs <= ATOL_MAX, f"{what}: max abs error {max_abs:.3e} > {ATOL_MAX}"
    assert worst <= REL_L2_ROW, f"{what}: worst row rel-L2 {worst:.3e} > {REL_L2_ROW} (row {int(rel.argmax())})"
    return max_abs, worst


class GpuBatch:
    """A workload's metadata and values on the GPU, plus the CPU copies the oracle reads."""

    def __init__(self, wl: W.PagedWorkload, vals: W.PagedValues, device="cuda"):
        self.wl = wl
        self.cpu = vals
        self.q = vals.q.to(device)
        self.k_new = vals.k_new.to(device)
        self.v_new = vals.v_new.to(device)
        self.k_cache = vals.k_cache.to(device)
        self.v_cache = vals.v_cache.to(device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.cu_q = torch.from_numpy(wl.cu_seqlens_q).to(device)
        self.cu_k = torch.from_numpy(wl.cu_seqlens_k).to(device)
        self.kv_lens = torch.from_numpy(wl.kv_lens).to(device)
        self.slots = torch.empty(wl.total_q, dtype=torch.int32, device=device)

    # ---- oracle side (CPU only) -------------------------------------------
    def oracle_slots(self) -> np.ndarray:
        return pa.slot_mapping(self.wl.q_lens, self.wl.kv_lens, self.wl.block_tables, self.wl.block_size)

    def oracle_pools(self):
        kc = f32(self.cpu.k_cache)
        vc = f32(self.cpu.v_cache)
        return pa.store_kvcache(kc, vc, f32(self.cpu.k_new), f32(self.cpu.v_new), self.oracle_slots(),
                                self.wl.block_size)

    def oracle_prefill(self, pools=None) -> np.ndarray:
        kc, vc = pools if pools is not None else self.oracle_pools()
        wl = self.wl
        return pa.prefill_varlen(f32(self.cpu.q), kc, vc, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.block_tables,
                                 wl.block_size, wl.softmax_scale)

    def oracle_decode(self, pools=None, rows=None) -> np.ndarray:
        kc, vc = pools if pools is not None else self.oracle_pools()
        wl = self.wl
        if rows is None:
            return pa.decode(f32(self.cpu.q), kc, vc, wl.block_tables, wl.kv_lens, wl.block_size, wl.softmax_scale)
        return pa.decode_rows(f32(self.cpu.q), kc, vc, wl.block_tables, wl.kv_lens, wl.block_size,
                              wl.softmax_scale, rows)

    # ---- CUDA side ---------------------------------------------------------
    def run_slots_and_store(self, pkv, decode: bool):
        wl = self.wl
        if decode:
            pkv.pkv_slot_mapping(self.block_tables, wl.num_blocks, wl.block_size, self.slots,
                                 context_lens=self.kv_lens)
        else:
            pkv.pkv_slot_mapping(self.block_tables, wl.num_blocks, wl.block_size, self.slots,
                                 cu_seqlens_q=self.cu_q, cu_seqlens_k=self.cu_k)
        pkv.pkv_store_kvcache(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache)

    def run_decode(self, pkv, out=None, workspace=None):
        wl = self.wl
        return pkv.pkv_decode(self.q, self.k_cache, self.v_cache, self.block_tables, self.kv_lens,
                              int(wl.kv_lens.max()), wl.softmax_scale, out=out, workspace=workspace)

    def run_prefill(self, pkv, out=None):
        wl = self.wl
        return pkv.pkv_prefill_varlen(self.q, self.k_cache, self.v_cache, self.cu_q, self.cu_k, self.block_tables,
                                      int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.softmax_scale, out=out)


def expect_no_device_error(pkv):
    code, info = pkv.pkv_get_device_error(clear=True)
    assert code == 0, f"device error {code} ({pkv.DEVERR.get(code)}), info {info}"


def check_sampler_ids(ids_gpu, logits, temps, seed, offset=0, max_near=2):
    """Sampled ids against the oracle's literal race on the same Philox noise."""
    lg = logits.cpu().double().numpy()
    T = temps.cpu().double().numpy()
    e = sm.exponential_noise(seed, offset, range(lg.shape[0]), lg.shape[1])
    ref, margin = sm.exponential_race(lg, T, e)
    got = ids_gpu.cpu().numpy()
    near = margin < NEAR_TIE
    assert np.array_equal(got[~near], ref[~near]), np.nonzero(got[~near] != ref[~near])
    for b in np.nonzero(near)[0]:
        z = lg[b] / T[b]
        r = np.exp(z - z.max()) / e[b]
        top2 = np.argsort(r)[-2:]
        assert got[b] in top2
    assert near.sum() <= max_near
    return int(near.sum())
