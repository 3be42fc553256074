"""The multi-device ring: one process per device, each holding one shard of the sequence.

Device i keeps its query shard Q_i and, at ring step r = 0..n-1, computes the block attention of
Q_i against the K/V block it holds -- that of shard j = (i - r) mod n -- folds it into its running
output, and meanwhile passes the block to device i + 1 and receives the next one from device i - 1
(LLM-101-CN "distributed hands-on code", section 6.2: block_attention, ring_send_recv_kv and
forward; airsota "M4-051 Ring Attention and sequence parallelism", section 3; "Lecture 30:
TP/PP/SP/CP", section 3.2).  The transfer of the next block runs while the current one is computed
(the questions after section 6.2 ask for exactly this overlap; M4-051's "communication overlap").
In the backward the K/V blocks go round again and the dK/dV accumulator of each block travels with
it: every device adds its contribution and passes it on, and after the n-th step the accumulator
arrives at the block's owner.

This module only schedules: every step of the arithmetic runs in the library's block calls
(ring_attn_block_fwd / ring_attn_block_bwd and their helpers, through ``ops``), and the blocks move
with torch.distributed point-to-point operations (NCCL between GPUs; gloo, staged through host
memory, in tests).

Shapes on device i: q, out, dout [B, H, S, d], k, v [B, Hkv, S, d], lse [B, H, S], with S = L / n
and n = world size; the rows are shard i's rows of the layout (contiguous, zigzag or striped), i.e.
rows [i*S, (i+1)*S) of the whole-sequence buffers of the single-device calls.
"""
from __future__ import annotations

import contextlib

import torch
import torch.distributed as dist


@contextlib.contextmanager
def _range(name):
    """An NVTX range (named step of the ring) for profilers that record them; free otherwise."""
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


class RingComm:
    """Point-to-point exchange with the ring neighbours: every call sends to rank + 1 and receives
    from rank - 1 (the direction of the pages' code, so that step r holds shard (rank - r) mod n).

    With the gloo backend and CUDA tensors the blocks are staged through host memory (gloo moves CPU
    tensors only); with NCCL they move device to device on NCCL's stream, ordered after the work
    already queued on the current stream, and ``wait`` orders the current stream after them."""

    def __init__(self, group=None):
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.next = (self.rank + 1) % self.world
        self.prev = (self.rank - 1) % self.world
        self.backend = dist.get_backend(group)
        self._gnext = dist.get_global_rank(group, self.next) if group is not None else self.next
        self._gprev = dist.get_global_rank(group, self.prev) if group is not None else self.prev

    def global_rank(self, r):
        """Global rank of rank r of this communicator's group."""
        return dist.get_global_rank(self.group, r) if self.group is not None else r

    def twin(self):
        """A second communicator over the same ranks, with the same rank numbering, created on first
        use (a collective call: every rank must reach it in the same order) and kept.  NCCL runs all
        point-to-point transfers of one communicator on one stream, one after the other; transfers
        on the twin run beside them, so a slow transfer on one does not hold back the other's.  Falls
        back to this communicator if the new group would number the ranks differently."""
        if getattr(self, "_twin", None) is None:
            ranks = [self.global_rank(r) for r in range(self.world)]
            group = dist.new_group(ranks=ranks, backend=self.backend)
            same = all(dist.get_group_rank(group, g) == r for r, g in enumerate(ranks))
            self._twin = RingComm(group) if same else self
        return self._twin

    def start(self, send, recv, tag=0, dst=None, src=None):
        """Starts sending the tensors `send` to rank dst (default rank + 1) and receiving into `recv`
        (same shapes and dtypes) from rank src (default rank - 1), ranks of this group, with message
        tags tag, tag + 1, ...: transfers that are in flight at the same time must use different
        tags.  Returns a handle for ``wait``."""
        gdst = self._gnext if dst is None else self.global_rank(dst)
        gsrc = self._gprev if src is None else self.global_rank(src)
        assert len(send) == len(recv)
        staged = self.backend == "gloo" and any(t.is_cuda for t in send)
        if staged:
            torch.cuda.current_stream().synchronize()  # the blocks to send are complete
            s_host = [t.cpu() for t in send]
            r_host = [torch.empty(t.shape, dtype=t.dtype) for t in recv]
        else:
            s_host, r_host = list(send), list(recv)
        ops = []
        for x, (s, r) in enumerate(zip(s_host, r_host)):
            ops.append(dist.P2POp(dist.isend, s, gdst, self.group, tag + x))
            ops.append(dist.P2POp(dist.irecv, r, gsrc, self.group, tag + x))
        works = dist.batch_isend_irecv(ops)
        return works, (r_host if staged else None), recv

    @staticmethod
    def wait(handle):
        """Completes a transfer: afterwards the received tensors may be read on the current stream."""
        works, r_host, recv = handle
        for w in works:
            w.wait()
        if r_host is not None:
            for dst, src in zip(recv, r_host):
                dst.copy_(src, non_blocking=False)


class LibraryOps:
    """The per-device compute of the ring: the library's block calls (CUDA)."""

    def __init__(self, stream=None):
        from . import binding

        self.b = binding
        self.stream = stream

    def empty_acc(self, shape, like):
        """A running-state or gradient accumulator (float32, on `like`'s device)."""
        return torch.empty(shape, dtype=torch.float32, device=like.device)

    def block_fwd(self, q, k, v, o_acc, lse_acc, n, i, j, accumulate, causal, layout):
        self.b.block_fwd(q, k, v, o_acc, lse_acc, n, i, j, accumulate, causal, layout, stream=self.stream)

    def convert(self, src, dtype):
        return self.b.f32_convert(src, dtype, stream=self.stream)

    def preprocess(self, out, dout):
        return self.b.bwd_preprocess(out, dout, stream=self.stream)

    def zero(self, x):
        self.b.f32_zero(x, stream=self.stream)

    def block_bwd(self, q, k, v, dout, lse, D, dq_acc, dk, dv, n, i, j, accumulate_kv, causal, layout):
        self.b.block_bwd(q, k, v, dout, lse, D, dq_acc, dk, dv, n, i, j, accumulate_kv, causal, layout,
                         stream=self.stream)

    def add(self, acc, part):
        self.b.f32_add(acc, part, stream=self.stream)


def ring_fwd(q, k, v, comm, causal=True, layout="zigzag", ops=None, keep_f32=False):
    """Ring forward on this device (rank i of n = world size): q [B,H,S,d] and k, v [B,Hkv,S,d] are
    shard i.  Returns (out [B,H,S,d] in q's dtype, lse [B,H,S] float32) for shard i's rows, and with
    keep_f32 also the float32 running output the out was converted from (for a backward's D)."""
    ops = ops or LibraryOps()
    n, i = comm.world, comm.rank
    B, H, S, d = q.shape
    o_acc = ops.empty_acc((B, H, S, d), q)
    lse_acc = ops.empty_acc((B, H, S), q)
    spare = _spare_blocks(k, v, n)
    cur = (k, v)
    for r in range(n):
        j = (i - r) % n
        # pass the block we hold on and take the next while this one is computed
        nxt = spare[r % 2] if r < n - 1 else None
        h = comm.start(cur, nxt) if nxt is not None else None
        with _range(f"ring fwd step {r}: block {j}"):
            ops.block_fwd(q, cur[0], cur[1], o_acc, lse_acc, n, i, j, r > 0, causal, layout)
        if h is not None:
            comm.wait(h)
            cur = nxt
    if keep_f32:
        return ops.convert(o_acc, q.dtype), lse_acc, o_acc
    return ops.convert(o_acc, q.dtype), lse_acc


def _spare_blocks(k, v, n):
    """The two receive slots of the K/V rotation.  A block is received into the slot that held the
    block of two steps before (computed and passed on by then), never into the caller's k and v."""
    return [(torch.empty_like(k), torch.empty_like(v)) for _ in range(min(2, n - 1))]


def ring_bwd(q, k, v, out, lse, dout, comm, causal=True, layout="zigzag", grad_dtype=torch.float32, ops=None):
    """Ring backward on this device: the inputs of ring_fwd plus its (out, lse) and the upstream
    gradient dout of shard i.  Returns (dq [B,H,S,d], dk, dv [B,Hkv,S,d]) of shard i in grad_dtype.
    out may be the float32 running output ring_fwd returns with keep_f32 (D from the unrounded output).

    Per step r (block j = (i - r) mod n): the K/V transfer of the next block starts, this device's
    contribution to block j's dK/dV is computed into `part` (dQ is added into the local dq_acc), the
    accumulator of block j arrives from device i - 1 (it holds the contributions of devices j .. i-1),
    `part` is added to it and it goes on to device i + 1.  After step n - 1 the accumulator that
    arrives is this device's own block, complete."""
    ops = ops or LibraryOps()
    n, i = comm.world, comm.rank
    B, H, S, d = q.shape
    Hkv = k.shape[1]
    D = ops.preprocess(out, dout)
    dq_acc = ops.empty_acc((B, H, S, d), q)
    ops.zero(dq_acc)
    kshape = (B, Hkv, S, d)
    acc = [tuple(ops.empty_acc(kshape, q) for _ in range(2)) for _ in range(2)]  # two accumulator slots
    part = tuple(ops.empty_acc(kshape, q) for _ in range(2)) if n > 1 else None
    spare = _spare_blocks(k, v, n)
    cur = (k, v)
    h_acc = None
    slot = 0
    for r in range(n):
        j = (i - r) % n
        nxt = spare[r % 2] if r < n - 1 else None
        h_kv = comm.start(cur, nxt) if nxt is not None else None
        with _range(f"ring bwd step {r}: block {j}"):
            # the first contribution to this device's own block starts its accumulator
            dst = acc[0] if r == 0 else part
            ops.block_bwd(q, cur[0], cur[1], dout, lse, D, dq_acc, dst[0], dst[1], n, i, j, False, causal, layout)
        if r > 0:
            comm.wait(h_acc)  # block j's accumulator from device i - 1, now in acc[slot]
            ops.add(acc[slot][0], part[0])
            ops.add(acc[slot][1], part[1])
        if n > 1:
            h_acc = comm.start(acc[slot], acc[1 - slot], tag=2)  # in flight with the K/V transfer
            slot = 1 - slot
        if h_kv is not None:
            comm.wait(h_kv)
            cur = nxt
    if n > 1:
        comm.wait(h_acc)  # this device's own block, with every device's contribution
    dk_acc, dv_acc = acc[slot]
    return ops.convert(dq_acc, grad_dtype), ops.convert(dk_acc, grad_dtype), ops.convert(dv_acc, grad_dtype)


# ------------------------------------------------------------------------------------------------
# Hierarchical ring: a local ring inside each group of devices, a global ring across the groups
# ------------------------------------------------------------------------------------------------
class RingGrid:
    """The ranks of a RingComm as `groups` groups of Q = world / groups consecutive ranks: rank
    r = p * Q + q is member q of group p.  The local ring runs inside a group (fast links, e.g. the
    devices of one node), the global ring across the groups at the same member index (the slow links
    between nodes): the hierarchical ring the pages suggest for very long contexts (agentalpha "Ring
    Attention vs tensor parallelism", follow-up 2).  Rank r still holds shard r.  Transfers between
    groups go over `gcomm`, the communicator's twin, so that they overlap the local ring's transfers
    instead of queueing with them."""

    def __init__(self, comm, groups):
        if groups < 1 or comm.world % groups:
            raise ValueError(f"{groups} groups do not divide {comm.world} ranks")
        self.comm = comm
        self.gcomm = comm.twin() if groups > 1 else comm
        self.P = groups
        self.Q = comm.world // groups
        self.p, self.q = divmod(comm.rank, self.Q)

    def rank(self, p, q):
        return (p % self.P) * self.Q + (q % self.Q)

    def held(self, a, b):
        """Shard of the K/V block this rank holds at global step a, local step b."""
        return self.rank(self.p - a, self.q - b)


def ring_fwd_2d(q, k, v, grid, causal=True, layout="zigzag", ops=None, keep_f32=False):
    """Ring forward over a RingGrid: for each global step a = 0..P-1 the block that arrived over the
    global ring (at a = 0 the device's own) goes round the local ring in Q local steps, while the next
    one comes from the previous group: one inter-group transfer per Q block steps, overlapped with
    them.  At (a, b) this rank holds the block of shard grid.held(a, b); over the P * Q steps it meets
    every shard once.  Same inputs and results as ring_fwd (keep_f32 as there)."""
    ops = ops or LibraryOps()
    comm, P, Q = grid.comm, grid.P, grid.Q
    n, i = comm.world, comm.rank
    B, H, S, d = q.shape
    o_acc = ops.empty_acc((B, H, S, d), q)
    lse_acc = ops.empty_acc((B, H, S), q)
    local_spare = _spare_blocks(k, v, Q)
    global_spare = _spare_blocks(k, v, P)
    origin = (k, v)
    step = 0
    for a in range(P):
        # this global step's block goes on to the next group while it circulates in this one
        h_g = (grid.gcomm.start(origin, global_spare[a % 2], tag=4, dst=grid.rank(grid.p + 1, grid.q),
                                src=grid.rank(grid.p - 1, grid.q)) if a < P - 1 else None)
        cur = origin
        for b in range(Q):
            nxt = local_spare[b % 2] if b < Q - 1 else None
            h_l = (comm.start(cur, nxt, tag=0, dst=grid.rank(grid.p, grid.q + 1), src=grid.rank(grid.p, grid.q - 1))
                   if nxt is not None else None)
            with _range(f"ring fwd step {a}.{b}: block {grid.held(a, b)}"):
                ops.block_fwd(q, cur[0], cur[1], o_acc, lse_acc, n, i, grid.held(a, b), step > 0, causal, layout)
            step += 1
            if h_l is not None:
                comm.wait(h_l)
                cur = nxt
        if h_g is not None:
            comm.wait(h_g)
            origin = global_spare[a % 2]
    if keep_f32:
        return ops.convert(o_acc, q.dtype), lse_acc, o_acc
    return ops.convert(o_acc, q.dtype), lse_acc


def ring_bwd_2d(q, k, v, out, lse, dout, grid, causal=True, layout="zigzag", grad_dtype=torch.float32, ops=None):
    """Ring backward over a RingGrid.  K/V move as in ring_fwd_2d; the dK/dV accumulator of a block
    always goes to the rank that holds that block next: the next member of the group inside a local
    round, the next member of the next group (one step along both rings) after its last local step,
    and after the last step of all to the block's owner.  Same inputs and results as ring_bwd."""
    ops = ops or LibraryOps()
    comm, P, Q = grid.comm, grid.P, grid.Q
    n, i = comm.world, comm.rank
    B, H, S, d = q.shape
    Hkv = k.shape[1]
    D = ops.preprocess(out, dout)
    dq_acc = ops.empty_acc((B, H, S, d), q)
    ops.zero(dq_acc)
    kshape = (B, Hkv, S, d)
    acc = [tuple(ops.empty_acc(kshape, q) for _ in range(2)) for _ in range(2)]
    part = tuple(ops.empty_acc(kshape, q) for _ in range(2)) if n > 1 else None
    local_spare = _spare_blocks(k, v, Q)
    global_spare = _spare_blocks(k, v, P)
    origin = (k, v)
    h_acc, slot, step = None, 0, 0
    for a in range(P):
        h_g = (grid.gcomm.start(origin, global_spare[a % 2], tag=4, dst=grid.rank(grid.p + 1, grid.q),
                                src=grid.rank(grid.p - 1, grid.q)) if a < P - 1 else None)
        cur = origin
        for b in range(Q):
            nxt = local_spare[b % 2] if b < Q - 1 else None
            h_l = (comm.start(cur, nxt, tag=0, dst=grid.rank(grid.p, grid.q + 1), src=grid.rank(grid.p, grid.q - 1))
                   if nxt is not None else None)
            j = grid.held(a, b)
            with _range(f"ring bwd step {a}.{b}: block {j}"):
                dst = acc[0] if step == 0 else part  # the first contribution starts the own block's accumulator
                ops.block_bwd(q, cur[0], cur[1], dout, lse, D, dq_acc, dst[0], dst[1], n, i, j, False, causal, layout)
            if step > 0:
                comm.wait(h_acc)  # block j's accumulator from its previous holder, now in acc[slot]
                ops.add(acc[slot][0], part[0])
                ops.add(acc[slot][1], part[1])
            if n > 1:
                if b < Q - 1:  # the next holder: the next member of this group
                    via, dst, src = comm, grid.rank(grid.p, grid.q + 1), grid.rank(grid.p, grid.q - 1)
                else:  # after a local round: the next member of the next group (between groups)
                    via, dst, src = grid.gcomm, grid.rank(grid.p + 1, grid.q + 1), grid.rank(grid.p - 1, grid.q - 1)
                h_acc = via.start(acc[slot], acc[1 - slot], tag=2, dst=dst, src=src)
                slot = 1 - slot
            step += 1
            if h_l is not None:
                comm.wait(h_l)
                cur = nxt
        if h_g is not None:
            comm.wait(h_g)
            origin = global_spare[a % 2]
    if n > 1:
        comm.wait(h_acc)  # this rank's own block, with every rank's contribution
    dk_acc, dv_acc = acc[slot]
    return ops.convert(dq_acc, grad_dtype), ops.convert(dk_acc, grad_dtype), ops.convert(dv_acc, grad_dtype)


# ------------------------------------------------------------------------------------------------
# The ring as a differentiable operation on each device
# ------------------------------------------------------------------------------------------------
class _DistributedRingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, comm, groups, causal, layout, ops, f32_out):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        if groups > 1:
            res = ring_fwd_2d(q, k, v, RingGrid(comm, groups), causal, layout, ops=ops, keep_f32=f32_out)
        else:
            res = ring_fwd(q, k, v, comm, causal, layout, ops=ops, keep_f32=f32_out)
        out, lse = res[0], res[1]
        ctx.save_for_backward(q, k, v, res[2] if f32_out else out, lse)
        ctx.cfg = (comm, groups, causal, layout, ops)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, saved, lse = ctx.saved_tensors
        comm, groups, causal, layout, ops = ctx.cfg
        dout = dout.contiguous()
        if groups > 1:
            grads = ring_bwd_2d(q, k, v, saved, lse, dout, RingGrid(comm, groups), causal, layout, q.dtype, ops=ops)
        else:
            grads = ring_bwd(q, k, v, saved, lse, dout, comm, causal, layout, q.dtype, ops=ops)
        return grads + (None,) * 6


def ring_attention_distributed(q, k, v, comm, causal=True, layout="zigzag", groups=1, ops=None, f32_out=False):
    """Ring attention on this device as a differentiable operation (the pages' RingAttention module,
    LLM-101-CN section 6.2): q [B,H,S,d], k, v [B,Hkv,S,d] are this rank's shard; the forward runs
    the ring (hierarchical with groups > 1) and the backward passes the blocks round again, so that
    every rank receives the gradients of its own shard.  Every rank of the communicator must call it
    with tensors of the same shapes.  f32_out: keep the float32 running output of the forward for the
    backward's D instead of the output rounded to q's dtype (twice the saved output's memory; closer
    to the exact gradient where a gradient is a short sum of large, cancelling terms)."""
    return _DistributedRingAttention.apply(q, k, v, comm, int(groups), causal, layout, ops or LibraryOps(),
                                           bool(f32_out))


class RingAttention(torch.nn.Module):
    """The pages' per-rank object (LLM-101-CN section 6.2): built from the model width ``dim``, the
    number of query heads, this rank and the world size; ``forward(Q, K, V)`` takes this rank's
    shard, Q [bs, heads, S, dim // heads] and K, V [bs, kv_heads, S, dim // heads], and returns this
    rank's rows of the output.  The scores are scaled by 1/sqrt(dim // heads), as on the page.

    Differences from the page's listing: the running maximum starts at minus infinity instead of
    -1e4 (so that no score is ever clipped), the transfers of the next block overlap the current
    block's work, K/V may have fewer heads than Q (grouped-query attention), and ``causal``,
    ``layout`` and ``groups`` select the causal mask, the shard layout and the hierarchical ring, and
    ``f32_out`` keeps the float32 output for the backward's D.
    The defaults are the page's: no mask, contiguous shards, one flat ring.  The output is
    differentiable; the backward passes the blocks round the ring again."""

    def __init__(self, dim, heads, rank=None, world_size=None, causal=False, layout="contiguous",
                 groups=1, group=None, ops=None, f32_out=False):
        super().__init__()
        if heads <= 0 or dim % heads:
            raise ValueError(f"dim {dim} is not a multiple of heads {heads}")
        self.dim, self.heads, self.head_dim = dim, heads, dim // heads
        self.comm = RingComm(group)
        if rank is not None and rank != self.comm.rank:
            raise ValueError(f"rank {rank} is not this process's rank {self.comm.rank} in the group")
        if world_size is not None and world_size != self.comm.world:
            raise ValueError(f"world_size {world_size} is not the group's size {self.comm.world}")
        self.rank, self.world_size = self.comm.rank, self.comm.world
        self.causal, self.layout, self.groups, self.ops, self.f32_out = causal, layout, int(groups), ops, f32_out

    def forward(self, Q, K, V):
        if Q.dim() != 4 or Q.shape[1] != self.heads or Q.shape[-1] != self.head_dim:
            raise ValueError(f"Q of shape {tuple(Q.shape)} is not [bs, {self.heads}, S, {self.head_dim}]")
        return ring_attention_distributed(Q, K, V, self.comm, self.causal, self.layout, self.groups, self.ops,
                                          self.f32_out)
