"""Seeded synthetic inputs for the MiTA forward operator.

This module holds no part of the operator's arithmetic: it only draws the
Q, K, V tensors (and names the shapes) that both the CUDA path and the CPU
oracle consume.  Every draw comes from ``torch.Generator('cpu')`` seeded per
workload, in a fixed order (centres -> cluster ids -> Q noise -> K noise ->
V), in fp32, rounded once to the workload's I/O type.

The workloads stand in for the vision and long-sequence settings the method
is evaluated on (DeiT-T / DeiT-S token grids of 14x14 with 5x5 landmarks,
a 56x56 high-resolution grid with 7x7 landmarks, a 64K-token 1-D sequence).
No dataset is used.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    gh: int          # token grid rows (1 for a 1-D sequence)
    gw: int          # token grid columns
    ph: int          # landmark grid rows
    pw: int          # landmark grid columns
    m: int
    k: int
    dtype: str       # "f32" or "bf16"
    gen: str         # "iid", "cluster_token", "cluster_patch", "cluster_span"
    centres: int = 0
    patch: int = 0   # cluster id fixed per patch x patch tile (cluster_patch)
    patch_offset: int = 0   # tiles start this many tokens before the grid's origin (cluster_patch)
    span: int = 0    # cluster id fixed per span of tokens (cluster_span)
    noise: float = 0.5
    seed: int = 1000

    @property
    def grid(self):
        return (self.gh, self.gw, self.ph, self.pw)

    @property
    def heads(self):
        return self.B * self.H

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads.  Seeds are 1000 + workload number.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 196, 64, 14, 14, 5, 5, 25, 25, "f32", "iid", seed=1001),
    "deit_t": Workload("deit_t", 128, 3, 196, 64, 14, 14, 5, 5, 25, 25, "bf16", "iid", seed=1002),
    "deit_s": Workload("deit_s", 256, 6, 196, 64, 14, 14, 5, 5, 25, 25, "bf16", "cluster_token",
                       centres=16, seed=1003),
    # 8 x 8 cluster tiles offset by 4 tokens from the 8 x 8 pooling bins, so
    # that related tokens are contiguous but not aligned with the landmarks
    "hires56": Workload("hires56", 16, 6, 3136, 64, 56, 56, 7, 7, 49, 64, "bf16", "cluster_patch",
                        centres=16, patch=8, patch_offset=4, seed=1004),
    "long1d": Workload("long1d", 2, 8, 65536, 128, 1, 65536, 1, 256, 256, 512, "bf16",
                       "cluster_span", centres=64, span=1024, seed=1005),
}


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def make_inputs(w: Workload, seed: int | None = None, return_ids: bool = False):
    """Q, K, V as contiguous CPU tensors [B, H, N, d] of the workload's type
    (and, with ``return_ids``, the cluster id of every token, [B, H, N])."""
    g = torch.Generator("cpu").manual_seed(w.seed if seed is None else seed)
    B, H, N, d = w.B, w.H, w.N, w.d
    ids = None
    if w.gen == "iid":
        Q = torch.randn(B, H, N, d, generator=g)
        K = torch.randn(B, H, N, d, generator=g)
    else:
        C = w.centres
        centres = torch.randn(B, H, C, d, generator=g)
        if w.gen == "cluster_token":
            ids = torch.randint(0, C, (B, H, N), generator=g)
        elif w.gen == "cluster_patch":
            # token (y, x) lies in tile ((y + o) // patch, (x + o) // patch)
            o = w.patch_offset
            ph_, pw_ = -(-(w.gh + o) // w.patch), -(-(w.gw + o) // w.patch)
            pid = torch.randint(0, C, (B, H, ph_, pw_), generator=g)
            ty = (torch.arange(w.gh) + o) // w.patch
            tx = (torch.arange(w.gw) + o) // w.patch
            ids = pid[:, :, ty][:, :, :, tx].reshape(B, H, N)
        elif w.gen == "cluster_span":
            sid = torch.randint(0, C, (B, H, N // w.span), generator=g)
            ids = sid.repeat_interleave(w.span, dim=2)
        else:
            raise ValueError(w.gen)
        base = torch.gather(centres, 2, ids.unsqueeze(-1).expand(B, H, N, d))
        Q = base + w.noise * torch.randn(B, H, N, d, generator=g)
        K = base + w.noise * torch.randn(B, H, N, d, generator=g)
    V = torch.randn(B, H, N, d, generator=g)
    dt = torch_dtype(w)
    out = Q.to(dt).contiguous(), K.to(dt).contiguous(), V.to(dt).contiguous()
    return out + (ids,) if return_ids else out


def make_integer_inputs(w: Workload, seed: int = 7):
    """Small-integer-valued Q, K, V for which every pooled mean is exactly
    representable in bf16 and every dot product is exact in fp32, so that
    expert indices and routes can be compared bit for bit.

    Bin token counts decide the value set of Q: 14x14 -> 5x5 bins hold 9, 12
    or 16 tokens, so Q takes values in 144*{-1,0,1} (integer means); 56x56 ->
    7x7 bins hold 64 tokens, so Q takes values in {-2..2} (means are
    multiples of 1/64 with at most 8 significant bits); 256-token 1-D bins
    take Q in {-1,0,1}.  Other grids fall back to {-1,0,1}.  K takes values
    in {-3..3}; V in {-4..4}/4.  Exact ties are frequent by construction.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    B, H, N, d = w.B, w.H, w.N, w.d
    if (w.gh, w.gw, w.ph, w.pw) == (14, 14, 5, 5):
        Q = 144.0 * torch.randint(-1, 2, (B, H, N, d), generator=g).float()
    elif (w.gh, w.gw, w.ph, w.pw) == (56, 56, 7, 7):
        Q = torch.randint(-2, 3, (B, H, N, d), generator=g).float()
    else:
        Q = torch.randint(-1, 2, (B, H, N, d), generator=g).float()
    K = torch.randint(-3, 4, (B, H, N, d), generator=g).float()
    V = torch.randint(-4, 5, (B, H, N, d), generator=g).float() / 4.0
    dt = torch_dtype(w)
    return Q.to(dt).contiguous(), K.to(dt).contiguous(), V.to(dt).contiguous()
