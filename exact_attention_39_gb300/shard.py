"""Data-parallel split of the forward over ranks, one GPU each.

Every (batch, head) problem of the forward is independent (the pages'
tiling works within one head), so G ranks each take a contiguous range of
the B*H problems and run ``fa_fwd`` on it by pointer offset: no data is
exchanged and no collective is needed.  Outputs stay sharded; a consumer
that needs them whole gathers them itself.
"""
import torch

from . import binding


def head_range(bh, world, rank):
    """The contiguous range [h0, h1) of the ``bh`` flattened (batch, head)
    problems that ``rank`` of ``world`` computes.  Ranges tile [0, bh) in
    rank order and their sizes differ by at most one; ranks past ``bh``
    get an empty range."""
    if bh < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("need bh >= 0, world >= 1 and 0 <= rank < world")
    base, extra = divmod(bh, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def fwd_shard(q, k, v, world, rank, causal=False, scale=None, stream=None,
              out=None, lse=None):
    """This rank's share of ``fwd(q, k, v)``: the problems ``head_range(B*H,
    world, rank)`` of the flattened batch and head axes, read in place from
    q [B, H, Nq, d] and k, v [B, H, Nk, d] (contiguous fp16/bf16 CUDA
    tensors).  Returns ``(o, lse, (h0, h1))`` with o [h1-h0, Nq, d] and lse
    [h1-h0, Nq] float32, equal to rows h0..h1-1 of the whole call's outputs
    flattened the same way.  ``out`` and ``lse``, when given, are written
    (contiguous tensors of those shapes)."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or k.shape[:2] != q.shape[:2]:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous (the shard is a pointer offset)")
    B, H, Nq, d = q.shape
    h0, h1 = head_range(B * H, world, rank)
    flat = lambda t: t.reshape(B * H, *t.shape[2:])
    # contiguous views of this rank's problems: their data pointers are the
    # offsets into the whole tensors
    q_r, k_r, v_r = (flat(t)[h0:h1].unsqueeze(0) for t in (q, k, v))
    if h1 == h0:
        o = q_r.new_empty((0, Nq, d)) if out is None else out
        lse = q_r.new_empty((0, Nq), dtype=torch.float32) if lse is None else lse
        return o, lse, (h0, h1)
    if out is not None and tuple(out.shape) != (h1 - h0, Nq, d):
        raise ValueError("out must be [h1 - h0, Nq, d]")
    if lse is not None and tuple(lse.shape) != (h1 - h0, Nq):
        raise ValueError("lse must be [h1 - h0, Nq]")
    o, l_ = binding.fwd(q_r, k_r, v_r, causal=causal, scale=scale, stream=stream,
                        out=None if out is None else out.unsqueeze(0),
                        lse=None if lse is None else lse.unsqueeze(0))
    return o[0], l_[0], (h0, h1)
