"""Test harness: run the CUDA library and the CPU oracle on the same seeded inputs.

The library side goes through the C ABI (decode_attention_rq_gb300); the oracle
side is oracle/.  The only thing they share is the input generator (synth).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import synth


@dataclasses.dataclass
class Case:
    L: int = 1
    P: int = 4
    G: int = 1
    H: int = 2
    d: int = 128
    g: int = 32
    B: int = 1
    Nmax: int = 256
    chained: bool = False
    seed: int = 0
    scaling: str = "ls"      # "ls" (least squares) or "norm" (norm ratio)
    rotation: str = "dense"  # "dense" (R as given) or "hadamard" (fast Walsh-Hadamard, no R on the device)
    Hq: int = 0              # query heads (0: = H, multi-head; else a multiple of H, grouped-query)

    def workload(self, anchor_is_base=True):
        alphas = synth.OURO_ALPHAS if self.P == 4 and anchor_is_base else tuple(
            [0.7, 0.85, 0.95, 1.0, 0.9, 0.8, 0.75, 0.7][: self.P] if self.P <= 8 else synth.group_alphas(self.P))
        return synth.Workload("case", self.L, self.P, self.G, self.H, self.d, self.g, self.B, self.Nmax,
                              alphas, anchor_is_base)


def rotation32(d, seed=0, kind="dense"):
    """The rotation as the device receives it (float32), and the same values in
    float64; for the Walsh-Hadamard mode the device gets none and the oracle
    takes H_d / sqrt(d)."""
    if kind == "hadamard":
        import oracle
        R = oracle.hadamard_matrix(d)
        return R.astype(np.float32), R
    R32 = synth.rotation(d, seed).astype(np.float32)
    return R32, R32.astype(np.float64)


class GpuCache:
    """A cache on the device driven through the C ABI."""

    def __init__(self, case: Case, R32: np.ndarray, device="cuda:0"):
        import decode_attention_rq_gb300 as rq
        self.rq = rq
        self.case = case
        self.device = device
        self.cfg = rq.rq_config(case.L, case.P, case.G, case.H, case.d, case.g, case.B, case.Nmax,
                                (rq.RQ_MODE_CHAINED if case.chained else rq.RQ_MODE_SHARED)
                                | (rq.RQ_MODE_NORM_RATIO if case.scaling == "norm" else 0)
                                | (rq.RQ_MODE_HADAMARD if case.rotation == "hadamard" else 0), case.Hq)
        self.nbytes = rq.rq_cache_bytes(self.cfg)
        assert self.nbytes > 0
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        self.R = None if case.rotation == "hadamard" else torch.from_numpy(R32).to(device)
        self.handle = rq.rq_cache_create(self.cfg, self.buf, self.nbytes, self.R)
        self.ws_bytes = rq.rq_decode_workspace_bytes(self.cfg, case.B)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.status = self.ws[:16].view(torch.int32)

    def close(self):
        if self.handle:
            self.rq.rq_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, layer, group, kv_bf16: torch.Tensor, start, batch=None):
        batch = self.case.B if batch is None else batch
        kv = kv_bf16.to(self.device).contiguous()
        sl = torch.as_tensor(np.asarray(start, dtype=np.int32), device=self.device)
        self.rq.rq_append(self.handle, layer, group, batch, kv, sl, kv.shape[-2], self.status)

    def decode(self, layer, group, loop, q, k_cur, v_cur, seq_lens, scale, batch=None):
        batch = self.case.B if batch is None else batch
        q = q.to(self.device).contiguous()
        k_cur = k_cur.to(self.device).contiguous()
        v_cur = v_cur.to(self.device).contiguous()
        sl = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device=self.device)
        out = torch.empty((batch, self.case.Hq or self.case.H, self.case.d), dtype=torch.float32, device=self.device)
        self.rq.rq_decode_attention(self.handle, layer, group, loop, batch, q, k_cur, v_cur, sl, scale,
                                    out, self.ws, self.ws_bytes)
        return out

    def decode_append(self, layer, group, q, kv_cur, seq_lens, scale, batch=None):
        """Anchor-loop call that also appends kv_cur ([P, 2, batch, H, d] or with a
        token axis of 1 before d) at position seq_lens[b]."""
        batch = self.case.B if batch is None else batch
        q = q.to(self.device).contiguous()
        kv = kv_cur.to(self.device).contiguous()
        sl = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device=self.device)
        out = torch.empty((batch, self.case.Hq or self.case.H, self.case.d), dtype=torch.float32, device=self.device)
        self.rq.rq_decode_attention_append(self.handle, layer, group, batch, q, kv, sl, scale, out, self.ws,
                                           self.ws_bytes)
        return out

    def bytes_host(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.buf.cpu().numpy()


def kv_for(case: Case, seed: int, ntok: int, anchor_is_base=True):
    return synth.looped_kv(seed, case.workload(anchor_is_base), batch=case.B, ntok=ntok)


def plane_views(buf: np.ndarray, geom, layer, group, b, h):
    """Slices of one region: dict name -> uint8 array (tile-major)."""
    base = geom.region_offset(layer, group, b, h)
    out = {"AK": buf[base + geom.anchor_plane(0): base + geom.anchor_plane(0) + geom.ntiles * geom.a_tile],
           "AV": buf[base + geom.anchor_plane(1): base + geom.anchor_plane(1) + geom.ntiles * geom.a_tile]}
    for j in range(geom.loops_per_group - 1):
        for kv, nm in ((0, "RK"), (1, "RV")):
            o = base + geom.res_plane(j, kv)
            out[f"{nm}{j}"] = buf[o: o + geom.ntiles * geom.r_tile]
    return out
