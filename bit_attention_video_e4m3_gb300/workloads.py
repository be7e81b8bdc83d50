"""Seeded synthetic inputs shaped like the pages' video-DiT attention workloads.

This module only draws random tensors and builds index structures; it holds
none of the method's arithmetic (no quantisation, no softmax).  The CUDA
path and the CPU oracle both receive what it produces.

Workloads (sequence lengths are latent grids frames x height x width):
  tiny       B=1, H=2,  T=1024, Q,K,V ~ N(0,1); identity permutation;
             exp2+cvt P-cast, S=256, forward.
  wan21      Wan2.1-1.3B-shaped dense: B=1, H=12, T=32760 (21x30x52).
             Q,K ~ N(0,1) plus constant per-channel offsets ~ N(0, 3^2) on 4
             seeded channels (same channels for every head, offsets drawn
             per (head, channel), independently for Q and K); V ~ N(0,1).
             exp2+cvt, S=256, no V-Smooth, forward.
  wan22      Wan2.2-14B-720p-shaped V-Smooth + ExpCast: B=1, H=40, T=75600
             (21x45x80).  Q,K ~ N(0,1).  V per head: 16 centres ~ N(0, 4^2)
             in R^128, a uniform cluster id per token (shuffled order),
             V = centre + 0.5 N(0, I); 0.5 % of each head's tokens have their
             row multiplied by 20.  Permutation = stable sort of tokens by
             cluster id.  ExpCast beta=-0.35, S=256.
  sta        sliding-tile sparse: B=1, H=24, grid 18x48x80 (T=69120), tiles of
             6x8x8 = 384 tokens stored tile-major; each query tile keeps the
             key tiles within an L-inf window of 3x5x5 tiles (|dt|<=1,
             |dh|<=2, |dw|<=2, clipped at the borders); Q,K,V ~ N(0,1).
  pcollapse  P-collapse stress: B=1, H=8, T=16384.  Channels 0..126 of Q and K
             ~ N(0,1)*sqrt(128/127); Q[...,127] = 4; the k_sink=4 keys at
             positions 0..3 have K[...,127] = Delta*sqrt(128)/4, all other keys
             K[...,127] = 0, so at scale 1/sqrt(128) the logits are ~N(0,1)
             plus Delta on the sinks.  Delta in {5..10}, forward/reverse,
             S in {1, 256, 448}.
  short4k    a single short head: B=1, H=1, T=4096, Q,K,V ~ N(0,1); exp2+cvt,
             S=256, no V-Smooth.  Its 32 query tiles leave most SMs idle: the
             case split-KV is for.

Seeds default to 1000 + workload index.  Tensors are bf16 [B, T, H, 128].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
KV_TILE = 128

WORKLOAD_ORDER = ["tiny", "wan21", "wan22", "sta", "pcollapse", "short4k"]

PCAST_EXP2_CVT = 0
PCAST_EXPCAST = 1


@dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    perm: torch.Tensor | None = None        # int32 [B, H, T]
    row_ptr: torch.Tensor | None = None     # int32 [nQt + 1]
    col: torch.Tensor | None = None         # int32 [nnz]
    vsmooth: bool = False
    pcast: int = PCAST_EXP2_CVT
    S: float = 256.0
    beta: float = -0.35
    reverse: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)

    def flops(self) -> float:
        """Algorithmic attention FLOPs: 4*B*H*T^2*d dense; kept tile pairs only when sparse."""
        if self.row_ptr is None:
            return 4.0 * self.B * self.H * self.T * self.T * HEAD_DIM
        rp = self.row_ptr.cpu().numpy()
        col = self.col.cpu().numpy()
        total = 0
        T = self.T
        for qt in range(len(rp) - 1):
            qrows = min(KV_TILE, T - qt * KV_TILE)
            for j in col[rp[qt]:rp[qt + 1]]:
                total += qrows * min(KV_TILE, T - int(j) * KV_TILE)
        return 4.0 * self.B * self.H * HEAD_DIM * total


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def sta_tile_lists(grid=(18, 48, 80), tile=(6, 8, 8), window=(3, 5, 5)):
    """CSR over 128-token tiles for sliding-tile attention on a tile-major token order.

    Query 3-D tile u keeps key 3-D tile v when |u_t - v_t| <= window_t // 2 in
    every axis (the L-inf window of the FPSAttention article, section 2.2),
    clipped at the grid border.  Each 3-D tile of 6*8*8 = 384 tokens spans
    three 128-token tiles; a query 128-tile inherits the list of its 3-D tile,
    expanded to 128-tiles and sorted ascending.
    """
    gt, gh, gw = (grid[i] // tile[i] for i in range(3))
    per3d = tile[0] * tile[1] * tile[2]
    assert per3d % KV_TILE == 0
    sub = per3d // KV_TILE
    half = [w // 2 for w in window]
    coords = [(a, b, c) for a in range(gt) for b in range(gh) for c in range(gw)]
    row_ptr = [0]
    col = []
    for (a, b, c) in coords:
        keep = []
        for v, (x, y, z) in enumerate(coords):
            if abs(a - x) <= half[0] and abs(b - y) <= half[1] and abs(c - z) <= half[2]:
                keep.extend(range(v * sub, v * sub + sub))
        keep.sort()
        for _ in range(sub):
            col.extend(keep)
            row_ptr.append(len(col))
    return np.asarray(row_ptr, dtype=np.int32), np.asarray(col, dtype=np.int32)


def make_workload(name: str, device="cpu", seed: int | None = None, T: int | None = None,
                  H: int | None = None, **over) -> Workload:
    """Build workload ``name``; T and H may be shrunk for small parity cases.

    Extra keyword overrides: delta (pcollapse), S, reverse, pcast, vsmooth.
    """
    idx = WORKLOAD_ORDER.index(name)
    seed = 1000 + idx if seed is None else seed
    g = _gen(device, seed)
    B = 1
    if name == "tiny":
        H = H or 2
        T = T or 1024
        q = _randn((B, T, H, HEAD_DIM), g, device)
        k = _randn((B, T, H, HEAD_DIM), g, device)
        v = _randn((B, T, H, HEAD_DIM), g, device)
        perm = torch.arange(T, device=device, dtype=torch.int32).expand(B, H, T).contiguous()
        w = Workload(name, B, T, H, q, k, v, perm=perm, vsmooth=over.get("vsmooth", True))
    elif name == "wan21":
        H = H or 12
        T = T or 32760
        q = _randn((B, T, H, HEAD_DIM), g, device)
        k = _randn((B, T, H, HEAD_DIM), g, device)
        v = _randn((B, T, H, HEAD_DIM), g, device)
        chans = torch.randperm(HEAD_DIM, generator=g, device=device)[:4]
        off_q = 3.0 * _randn((H, 4), g, device)
        off_k = 3.0 * _randn((H, 4), g, device)
        q[:, :, :, chans] += off_q[None, None]
        k[:, :, :, chans] += off_k[None, None]
        w = Workload(name, B, T, H, q, k, v, vsmooth=over.get("vsmooth", False))
        w.extra["offset_channels"] = chans.cpu().tolist()
    elif name == "wan22":
        H = H or 40
        T = T or 75600
        q = _randn((B, T, H, HEAD_DIM), g, device)
        k = _randn((B, T, H, HEAD_DIM), g, device)
        centres = 4.0 * _randn((H, 16, HEAD_DIM), g, device)
        cid = torch.randint(0, 16, (H, T), generator=g, device=device)
        v = torch.empty((B, T, H, HEAD_DIM), device=device, dtype=torch.float32)
        n_out = int(round(0.005 * T))
        perm = torch.empty((B, H, T), device=device, dtype=torch.int32)
        for h in range(H):
            vh = centres[h][cid[h]] + 0.5 * _randn((T, HEAD_DIM), g, device)
            outl = torch.randperm(T, generator=g, device=device)[:n_out]
            vh[outl] *= 20.0
            v[0, :, h, :] = vh
            perm[0, h] = torch.sort(cid[h], stable=True).indices.to(torch.int32)
        w = Workload(name, B, T, H, q, k, v, perm=perm, vsmooth=over.get("vsmooth", True),
                     pcast=over.get("pcast", PCAST_EXPCAST))
    elif name == "sta":
        H = H or 24
        grid = over.get("grid", (18, 48, 80))
        T_full = grid[0] * grid[1] * grid[2]
        T = T_full
        q = _randn((B, T, H, HEAD_DIM), g, device)
        k = _randn((B, T, H, HEAD_DIM), g, device)
        v = _randn((B, T, H, HEAD_DIM), g, device)
        rp, cl = sta_tile_lists(grid=grid)
        w = Workload(name, B, T, H, q, k, v,
                     row_ptr=torch.from_numpy(rp).to(device), col=torch.from_numpy(cl).to(device),
                     vsmooth=over.get("vsmooth", False))
    elif name == "short4k":
        H = H or 1
        T = T or 4096
        q = _randn((B, T, H, HEAD_DIM), g, device)
        k = _randn((B, T, H, HEAD_DIM), g, device)
        v = _randn((B, T, H, HEAD_DIM), g, device)
        w = Workload(name, B, T, H, q, k, v, vsmooth=over.get("vsmooth", False))
    elif name == "pcollapse":
        H = H or 8
        T = T or 16384
        delta = float(over.get("delta", 7.0))
        sc = math.sqrt(128.0 / 127.0)
        q = _randn((B, T, H, HEAD_DIM), g, device) * sc
        k = _randn((B, T, H, HEAD_DIM), g, device) * sc
        v = _randn((B, T, H, HEAD_DIM), g, device)
        q[..., 127] = 4.0
        k[..., 127] = 0.0
        k[:, 0:4, :, 127] = delta * math.sqrt(128.0) / 4.0
        w = Workload(name, B, T, H, q, k, v, vsmooth=over.get("vsmooth", False),
                     S=float(over.get("S", 256.0)), reverse=bool(over.get("reverse", False)))
        w.extra["delta"] = delta
    else:
        raise KeyError(name)
    w.q = w.q.to(torch.bfloat16).contiguous()
    w.k = w.k.to(torch.bfloat16).contiguous()
    w.v = w.v.to(torch.bfloat16).contiguous()
    for key in ("S", "reverse", "pcast", "beta"):
        if key in over and name not in ("pcollapse",):
            setattr(w, key, over[key])
    w.seed = seed
    return w


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a bf16 tensor's bits (copied to host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
