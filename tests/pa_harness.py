"""Runs one workload step through the CUDA library and through the oracle.

The two sides share only the seeded inputs from `workloads`: the oracle receives host
copies of the inputs taken before any library call, and computes its own slot mapping,
cache write, block copies and attention.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of `dtype` at |ref| (normal range)."""
    mant = {"f16": 10, "bf16": 7, "f32": 23}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14)))
    return 2.0 ** (e - mant - 1)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class StepRun:
    """Device copies of a step's inputs plus the library calls of one step."""

    def __init__(self, step: W.Step, device="cuda"):
        self.step = step
        self.device = device
        self.vals = W.make_values(step, device)
        self.meta = {}
        for kind in ("decode", "prefill"):
            b = getattr(step, kind)
            if b is None:
                continue
            self.meta[kind] = {
                "bt": torch.from_numpy(b.block_tables).to(device),
                "ctx": torch.from_numpy(b.context_lens).to(device),
                "cu": torch.from_numpy(b.cu_q_lens).to(device),
            }
        self.pairs = (torch.from_numpy(step.cow_pairs).to(device)
                      if step.cow_pairs is not None else None)

    # ------------------------------------------------------------------ host inputs
    def host_pool(self, block_ids: Optional[np.ndarray] = None):
        """Host copies of the pool (all of it, or only `block_ids`), before the step."""
        kc, vc = self.vals["k_cache"], self.vals["v_cache"]
        if block_ids is None:
            return W.to_numpy(kc), W.to_numpy(vc)
        idx = torch.from_numpy(np.asarray(block_ids, dtype=np.int64)).to(kc.device)
        return W.to_numpy(kc.index_select(0, idx)), W.to_numpy(vc.index_select(0, idx))

    def host_values(self):
        return {k: W.to_numpy(v) for k, v in self.vals.items()
                if k not in ("k_cache", "v_cache")}

    # ------------------------------------------------------------------ library calls
    def run(self, out_dtype: Optional[torch.dtype] = torch.float32, kinds=("decode", "prefill"),
            share_prefix: bool = False):
        import paged_kv_cache_53_gb300 as pa
        st, sh = self.step, self.step.shape
        kc, vc = self.vals["k_cache"], self.vals["v_cache"]
        res: Dict[str, torch.Tensor] = {}
        if self.pairs is not None:
            pa.copy_blocks([kc], [vc], self.pairs)
        for kind, m in self.meta.items():
            b = getattr(st, kind)
            slots = torch.empty(b.num_new_tokens, dtype=torch.int64, device=self.device)
            pa.slot_mapping(slots, m["bt"], m["cu"], m["ctx"], sh.block_size, st.num_blocks)
            pa.reshape_and_cache(self.vals[f"k_new_{kind}"], self.vals[f"v_new_{kind}"], kc, vc,
                                 slots)
            res[f"slots_{kind}"] = slots
        if "decode" in self.meta and "decode" in kinds:
            b, m = st.decode, self.meta["decode"]
            od = out_dtype or kc.dtype
            out = torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), dtype=od,
                              device=self.device)
            if share_prefix:
                blocks, plen, sharers = st.shared_prefix
                nbytes = pa.decode_shared_prefix_workspace_bytes(
                    b.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, b.max_ctx,
                    sh.block_size, len(sharers), plen)
                ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
                pa.decode_shared_prefix(out, self.vals["q_decode"], kc, vc, m["bt"], m["ctx"],
                                        b.max_ctx, torch.from_numpy(blocks).to(self.device),
                                        plen, torch.from_numpy(sharers).to(self.device),
                                        st.scale, ws)
            else:
                ws = torch.empty(pa.decode_workspace_bytes(b.num_seqs, sh.num_q_heads,
                                                           sh.num_kv_heads, sh.head_dim,
                                                           b.max_ctx, sh.block_size),
                                 dtype=torch.uint8, device=self.device)
                pa.decode(out, self.vals["q_decode"], kc, vc, m["bt"], m["ctx"], b.max_ctx,
                          st.scale, ws)
            res["out_decode"] = out
        if "prefill" in self.meta and "prefill" in kinds:
            b, m = st.prefill, self.meta["prefill"]
            od = out_dtype or kc.dtype
            out = torch.empty((b.num_new_tokens, sh.num_q_heads, sh.head_dim), dtype=od,
                              device=self.device)
            nbytes = pa.prefill_workspace_bytes(b.num_seqs, b.num_new_tokens, b.max_q,
                                                sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                                                b.max_ctx, sh.block_size)
            ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.device)
            pa.prefill_chunk(out, self.vals["q_prefill"], kc, vc, m["bt"], m["cu"], m["ctx"],
                             b.max_q, b.max_ctx, st.scale, ws)
            res["out_prefill"] = out
        torch.cuda.synchronize()
        return res


# ---------------------------------------------------------------------- oracle side
def oracle_step(step: W.Step, kc: np.ndarray, vc: np.ndarray, vals: Dict[str, np.ndarray],
                decode_seqs: Optional[Sequence[int]] = None,
                prefill_tokens: Optional[Sequence[int]] = None,
                block_map: Optional[np.ndarray] = None):
    """The oracle's version of one step on host arrays (modified in place).

    With `block_map` the pool arrays hold only some physical blocks: block_map[i] is the
    physical id of row i, and tables are renumbered to rows before the oracle walks them.
    """
    sh = step.shape
    out = {}

    def remap(tables):
        if block_map is None:
            return tables
        lut = {int(p): i for i, p in enumerate(block_map)}
        return np.vectorize(lambda x: lut.get(int(x), -1), otypes=[np.int32])(tables)

    if step.cow_pairs is not None:
        pairs = step.cow_pairs
        if block_map is not None:
            pairs = remap(pairs)
            pairs = pairs[(pairs >= 0).all(axis=1)]
        oracle.copy_blocks([kc, vc], pairs)
    for kind in ("decode", "prefill"):
        b = getattr(step, kind)
        if b is None:
            continue
        slots = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, sh.block_size)
        out[f"slots_{kind}"] = slots
        write = slots
        if block_map is not None:
            blk, off = np.divmod(slots, sh.block_size)
            lut = {int(p): i for i, p in enumerate(block_map)}
            rows = np.array([lut.get(int(x), -1) for x in blk], dtype=np.int64)
            write = np.where(rows >= 0, rows * sh.block_size + off, -1)
        oracle.reshape_and_cache(vals[f"k_new_{kind}"], vals[f"v_new_{kind}"], kc, vc, write)
    if step.decode is not None:
        b = step.decode
        seqs = range(b.num_seqs) if decode_seqs is None else decode_seqs
        out["out_decode"] = oracle.decode_attention_rows(
            vals["q_decode"], kc, vc, remap(b.block_tables), b.context_lens, step.scale, sh.dtype,
            list(seqs))
    if step.prefill is not None:
        b = step.prefill
        toks = range(b.num_new_tokens) if prefill_tokens is None else prefill_tokens
        out["out_prefill"] = oracle.prefill_chunk_attention_rows(
            vals["q_prefill"], kc, vc, remap(b.block_tables), b.cu_q_lens, b.context_lens,
            step.scale, sh.dtype, list(toks))
    return out


def blocks_of(batch: W.Batch, seqs: Sequence[int], block_size: int) -> np.ndarray:
    """Physical blocks the listed sequences use."""
    ids = []
    for s in seqs:
        n = oracle.blocks_for_tokens(int(batch.context_lens[s]), block_size)
        ids.extend(batch.block_tables[s, :n].tolist())
    return np.unique(np.asarray(ids, dtype=np.int64))


def max_abs_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
