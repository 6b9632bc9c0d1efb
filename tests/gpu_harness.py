"""Helpers for the GPU parity tests: put a workload on the device, run one step
through the library, and check it against the CPU oracle.

The oracle and the library get the same seeded arrays from ``workloads``;
nothing the oracle consumes comes from the library's output.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_156_gb300 as pkv
import workloads as W

TORCH_DT = {W.F16: torch.float16, W.BF16: torch.bfloat16}
# max-abs-error bounds for attention outputs on N(0,1) inputs, fp32 accumulation
TOL = {W.F16: 2e-3, W.BF16: 1e-2}


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DT[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceStep:
    """One decode step of a workload, resident on the device."""

    def __init__(self, wl: W.Workload, pools: str = "host", device="cuda", partition_tokens: int = 0):
        s = wl.spec
        self.wl = wl
        self.dt = s.dtype
        self.q = to_dev(wl.q, s.dtype, device)
        self.k_new = to_dev(wl.k_new, s.dtype, device)
        self.v_new = to_dev(wl.v_new, s.dtype, device)
        self.slot_mapping = torch.from_numpy(wl.slot_mapping).to(device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.copy_pairs = torch.from_numpy(wl.copy_pairs).to(device)
        if pools == "host":
            self.kc = [to_dev(x, s.dtype, device) for x in wl.key_caches]
            self.vc = [to_dev(x, s.dtype, device) for x in wl.value_caches]
        else:
            self.kc, self.vc = [], []
            for l in range(s.num_layers):
                k, v = W.device_pools(wl, l, device)
                self.kc.append(k)
                self.vc.append(v)
        self.out = [torch.empty_like(self.q) for _ in range(s.num_layers)]
        self.partition_tokens = partition_tokens
        self.workspace = pkv.alloc_workspace(s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, wl.max_seq_len,
                                             partition_tokens, device)

    def run(self):
        """copy-on-write copies, then per layer: append, decode."""
        if self.copy_pairs.shape[0]:
            pkv.copy_blocks(self.kc, self.vc, self.copy_pairs)
        for l in range(len(self.kc)):
            pkv.paged_kv_append(self.k_new, self.v_new, self.kc[l], self.vc[l], self.slot_mapping)
            self.decode(l)

    def run_planned_fused(self, inputs_ready=False):
        """The benchmark's step: copy-on-write copies, one plan for the step, then per layer
        the slot write fused into the decode launch (one new token per sequence); with
        ``inputs_ready``, every layer after the first starts its tile loads early, as the
        benchmark's step does."""
        wl, s = self.wl, self.wl.spec
        assert wl.num_tokens == s.num_seqs, "the fused call writes one token per sequence"
        if self.copy_pairs.shape[0]:
            pkv.copy_blocks(self.kc, self.vc, self.copy_pairs)
        total = int(wl.seq_lens.sum())
        pkv.decode_plan(self.workspace, self.block_tables, self.seq_lens, s.num_heads, self.kc[0], wl.max_seq_len,
                        self.partition_tokens, sum_seq_lens=total)
        for l in range(len(self.kc)):
            pkv.paged_kv_append_decode(self.out[l], self.q, self.k_new, self.v_new, self.kc[l], self.vc[l],
                                       self.slot_mapping, self.block_tables, self.seq_lens, wl.scale,
                                       max_seq_len=wl.max_seq_len, workspace=self.workspace,
                                       partition_tokens=self.partition_tokens, planned=True, sum_seq_lens=total,
                                       inputs_ready=inputs_ready and l > 0)

    def decode(self, l=0):
        wl = self.wl
        pkv.paged_attention_decode(self.out[l], self.q, self.kc[l], self.vc[l], self.block_tables, self.seq_lens,
                                   wl.scale, max_seq_len=wl.max_seq_len, workspace=self.workspace,
                                   partition_tokens=self.partition_tokens)


def oracle_caches_after_step(wl: W.Workload, kc_bits: np.ndarray, vc_bits: np.ndarray):
    """The oracle's view of one layer's pools after the step's copies and slot writes."""
    kc, vc = kc_bits.copy(), vc_bits.copy()
    if len(wl.copy_pairs):
        oracle.copy_blocks_ref([kc], [vc], wl.copy_pairs)
    oracle.append_ref(kc, vc, wl.k_new, wl.v_new, wl.slot_mapping)
    return kc, vc


def oracle_attention(wl: W.Workload, kc: np.ndarray, vc: np.ndarray, seqs=None) -> np.ndarray:
    seqs = np.arange(wl.spec.num_seqs) if seqs is None else np.asarray(seqs)
    return oracle.attention_ref(wl.q[seqs], kc, vc, wl.block_tables[seqs], wl.seq_lens[seqs], wl.scale,
                                wl.spec.num_kv_heads, wl.spec.dtype)


def mean_abs_err(gpu_out: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    return float(np.mean(np.abs(g - ref))) if g.size else 0.0


def max_abs_err(gpu_out: torch.Tensor, ref: np.ndarray, seqs=None) -> float:
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    if seqs is not None:
        g = g[np.asarray(seqs)]
    return float(np.max(np.abs(g - ref))) if g.size else 0.0
