"""The fused step across tensor-parallel ranks, split at token boundaries.

[W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
Arithmetic, Not Finer Tiles", section "Fix two: RMSNorm was never
insignificant": the all-reduce after a row-parallel projection is taken apart
into a reduce-scatter and an all-gather at token boundaries, so that each rank
normalises only its own whole token rows instead of every rank normalising the
whole batch.

Each rank holds its own [T, H] partial (its projection output), the [T, H]
residual (the same on every rank) and gamma. One call of ``TokenShardStep``:

1. all-to-all: rank j sends the rows of rank r's shard of its partial to rank
   r (``tw_shard_rows``: contiguous shards of ceil(T / W) rows in rank order).
   Rank r receives W slices of its shard, slice j from rank j. This moves the
   same bytes as a reduce-scatter but leaves the reduction to step 2.
2. the fused step (``tw_fused_reduce_residual_rmsnorm``) on the rank's shard
   with N = W partials, the received slices in rank order: the sum runs in
   fp32 in rank order inside the kernel, so the shard's rows are bitwise the
   rows of the one-GPU step over all W partials.
3. all-gather of the shard's output and updated residual, so every rank ends
   with the whole [T, H] output and residual.

Collectives are torch.distributed's (NCCL between GPUs); the reduction and
the norm run in libtw's kernel. No multicast memory and no peer pointer is
handed to a kernel. Argument marshalling only: this module computes nothing
itself.
"""

import reduce_rmsnorm_gb300 as tw


class TokenShardStep:
    """The token-shard step for a fixed [T, H] on one rank of ``group``.

    Buffers for the received slices and the gathered pieces are allocated
    once, at construction, on ``device``. ``local_step`` is the call that runs
    step 2; it defaults to the libtw fused step and takes
    ``(partials [W, rows, H], residual [rows, H] in/out, gamma, eps,
    out [rows, H])``.
    """

    def __init__(self, T, H, group=None, device=None, dtype=None, local_step=None):
        import torch
        import torch.distributed as dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if self.world > tw.TW_MAX_PARTIALS:
            raise ValueError("at most %d ranks: each rank's shard sums one partial per rank"
                             % tw.TW_MAX_PARTIALS)
        self.T, self.H = int(T), int(H)
        self.shards = [tw.tw_shard_rows(self.T, self.world, r) for r in range(self.world)]
        self.row0, self.rows = self.shards[self.rank]
        self.s = -(-self.T // self.world) if self.T else 0  # padded shard rows
        dtype = dtype or torch.bfloat16
        kw = dict(dtype=dtype, device=device)
        self.recv = torch.empty((self.world, self.rows, self.H), **kw)
        self.y_piece = torch.zeros((self.s, self.H), **kw)
        self.r_piece = torch.zeros((self.s, self.H), **kw)
        self.exact = self.world * self.s == self.T  # pieces tile the batch with no padding
        if not self.exact:
            self.y_all = torch.empty((self.world * self.s, self.H), **kw)
            self.r_all = torch.empty((self.world * self.s, self.H), **kw)
        self.local_step = local_step or self._fused

    @staticmethod
    def _fused(partials, residual, gamma, eps, out):
        tw.tw_fused_reduce_residual_rmsnorm(partials, residual, gamma, eps, out)

    def __call__(self, partial, residual, gamma, eps, out):
        """partial: this rank's [T, H]; residual: [T, H], updated in place on
        every rank; out: [T, H], written on every rank."""
        import torch.distributed as dist
        T, H = self.T, self.H
        for name, t in (("partial", partial), ("residual", residual), ("out", out)):
            if tuple(t.shape) != (T, H) or not t.is_contiguous():
                raise ValueError("%s must be a contiguous [%d, %d] tensor" % (name, T, H))
        if T == 0:
            return
        sizes = [rows * H for _, rows in self.shards]
        dist.all_to_all_single(self.recv.view(-1), partial.view(-1),
                               output_split_sizes=[self.rows * H] * self.world,
                               input_split_sizes=sizes, group=self.group)
        a, n = self.row0, self.rows
        if n > 0:
            self.r_piece[:n].copy_(residual[a:a + n])
            self.local_step(self.recv, self.r_piece[:n], gamma, eps, self.y_piece[:n])
        if self.exact:
            dist.all_gather_into_tensor(out, self.y_piece, group=self.group)
            dist.all_gather_into_tensor(residual, self.r_piece, group=self.group)
        else:
            dist.all_gather_into_tensor(self.y_all, self.y_piece, group=self.group)
            dist.all_gather_into_tensor(self.r_all, self.r_piece, group=self.group)
            out.copy_(self.y_all[:T])
            residual.copy_(self.r_all[:T])
