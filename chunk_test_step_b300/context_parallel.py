"""Context-parallel chunk update: one large update chunk cut across ranks by tokens.

The LaCT review page, section "Video and distributed computation", scales a
chunk past one device this way: the chunk's tokens are split among the
devices, each device computes the update gradients of its own slice, the
gradients are combined, and every device applies the one resulting update
(the pages report 1-3 % overhead for it).

Why the combine is exact. The chunk gradient of
L = -sum_i eta_i <f_W(k_i), v_i> is a sum over the chunk's tokens, so the sum
over ranks of the slice gradients is the whole chunk's gradient (up to the
order of the additions). The update rule (GD, momentum or Muon) and the row
renorm then run on every rank from that same sum, so the fast weights stay
identical everywhere with no further exchange; queries can be read on any
rank.

Exchange: one all-reduce (sum) per chunk of the three gradient matrices,
3 * d * dh fp32 per (b, h) (12 * d * dh bytes: 6.3 MB for 8 heads of d = 128,
dh = 512), or d * d for the linear memory.

On each rank the gradient and the update are liblact calls
(lact_chunk_gradient, lact_apply_gradient); this module cuts the tokens, owns
the gradient buffer and issues the collective through torch.distributed (NCCL
between GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch

from . import lact as L

TILE = 128   # tokens per gradient tile of the tensor-core kernels


def token_range(n_tok: int, rank: int, world: int, tile: int = TILE) -> tuple[int, int]:
    """Tokens [start, stop) of `rank`'s slice of an n_tok-token chunk.

    Slices are contiguous and hold whole tiles of `tile` tokens, balanced to
    within one tile (the first ranks take the extra tiles); only the slice
    holding the chunk's end can be ragged. Ranks beyond the last tile get an
    empty slice.
    """
    if world < 1 or not 0 <= rank < world or n_tok < 0 or tile < 1:
        raise ValueError((n_tok, rank, world, tile))
    tiles = -(-n_tok // tile)
    base, extra = divmod(tiles, world)
    t0 = rank * base + min(rank, extra)
    t1 = t0 + base + (1 if rank < extra else 0)
    return min(n_tok, t0 * tile), min(n_tok, t1 * tile)


class GradientBuffer:
    """dL/dW1, dL/dW2, dL/dW3 of every (b, h) as views of one flat fp32 tensor,
    so that a single collective carries them (the linear memory: one matrix)."""

    def __init__(self, B: int, H: int, d: int, dh: int, linear: bool, device, dtype=torch.float32):
        shapes = ((d, d),) if linear else ((dh, d), (d, dh), (dh, d))
        sizes = [B * H * a * b for a, b in shapes]
        self.flat = torch.zeros(sum(sizes), dtype=dtype, device=device)
        self.mats = []
        off = 0
        for (a, b), n in zip(shapes, sizes):
            self.mats.append(self.flat[off:off + n].view(B, H, a, b))
            off += n

    def views(self):
        """The matrices in the C ABI's argument order, None for absent ones."""
        return self.mats + [None] * (3 - len(self.mats))

    @property
    def nbytes(self) -> int:
        return self.flat.numel() * self.flat.element_size()


class ContextParallelUpdate:
    """One fast-weight state per rank, updated from a token slice per rank.

    `layer` is the rank's state (a LactLayer, or anything with `cfg` and
    `handle`); every rank starts from the same weights. `group` is the
    torch.distributed group of the ranks sharing the chunk (None: the default
    group if one is initialised, else a single rank). `gradient` and `step`
    replace the two liblact calls (signatures as `lact_gradient` and
    `lact_step` below); the tests use this to run the same composition with
    the CPU oracle. The gradient buffer is fp32, the C ABI's gradient type
    (`dtype` changes it for such replacements).
    """

    def __init__(self, layer, group=None, device=None, gradient=None, step=None, dtype=torch.float32):
        import torch.distributed as dist
        self.layer = layer
        self.group = group
        if dist.is_available() and dist.is_initialized():
            self.rank, self.world = dist.get_rank(group), dist.get_world_size(group)
        else:
            self.rank, self.world = 0, 1
        c = layer.cfg
        if device is None:
            device = getattr(getattr(layer, "workspace", None), "device", "cuda")
        self.buf = GradientBuffer(c.B, c.H, c.d, c.dh, c.memory == L.LACT_MEM_LINEAR, device, dtype)
        self._gradient = gradient or self.lact_gradient
        self._step = step or self.lact_step

    # ---- the liblact calls of each phase
    def lact_gradient(self, k, v, eta, n_tok: int, grads, stream=None) -> None:
        L.lact_chunk_gradient(self.layer.handle, k, v, eta, n_tok, *grads, stream)

    def lact_step(self, grads, stream=None) -> None:
        L.lact_apply_gradient(self.layer.handle, *grads, stream)

    # ---- phases
    def slice(self, n_tok: int) -> tuple[int, int]:
        """This rank's tokens of an n_tok-token chunk."""
        return token_range(n_tok, self.rank, self.world)

    def compute_gradient(self, k, v, eta, n_local: int, stream=None) -> None:
        """Gradient of this rank's slice ([B, H, n_local, d] k, v; [B, H, n_local]
        eta) into the buffer; an empty slice contributes zeros."""
        self._gradient(k, v, eta, n_local, self.buf.views(), stream)

    def combine(self, stream=None) -> None:
        """Sum the buffers of all ranks (one all-reduce), in place."""
        if self.world == 1:
            return
        import torch.distributed as dist
        if stream is not None and self.buf.flat.is_cuda:
            with torch.cuda.stream(stream):
                dist.all_reduce(self.buf.flat, op=dist.ReduceOp.SUM, group=self.group)
        else:
            dist.all_reduce(self.buf.flat, op=dist.ReduceOp.SUM, group=self.group)

    def step(self, stream=None) -> None:
        """The update rule + row renorm from the combined gradient."""
        self._step(self.buf.views(), stream)

    def update(self, k, v, eta, n_local: int, stream=None) -> None:
        """One update of the whole chunk from this rank's slice of it."""
        self.compute_gradient(k, v, eta, n_local, stream)
        self.combine(stream)
        self.step(stream)
