"""Context-parallel prefill: one packed batch split over ranks by tokens.

The pages run the layer under context parallelism, where the token dimension
of a packed batch is cut into consecutive slices, one per rank ("[Qwen3.5 MoE]
Add hybrid decoder model (GatedDeltaNet + full attention + MoE)", Summary:
parallelize.py bullet, TP/FSDP/CP/EP; "feat(models): dense Qwen3.5 custom
attention", Summary: ring / Ulysses CP substitution, and its E2E notes: CP at
cp = 2).  For attention that is a ring of key/value exchanges; for this layer
the only quantity that crosses a slice boundary inside a sequence is what the
recurrence and the width-4 causal conv carry: the fp32 state of every value
head and the raw inputs of the last three tokens (the conv history).

Rank r holds tokens [t0_r, t1_r) of the batch.  A sequence that starts before
t0_r continues on rank r from the state and conv history rank r - 1 leaves it
with; rank r runs its slice with ``gdn_prefill_carry`` (each local sequence
from its own initial state, the continued one from the received state and
conv history) and hands the state and conv history of a sequence that goes on
past t1_r to rank r + 1.  This is the sequential state hand-off: a rank whose
slice starts inside a sequence waits for its predecessor.  The host logic here
only plans the slices and moves the carried tensors (torch.distributed
point-to-point, one send and one receive per boundary); every step of the
layer runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

__all__ = ["RankPlan", "plan_rank", "context_parallel_prefill"]


@dataclass(frozen=True)
class RankPlan:
    """The part of a packed batch one rank computes."""
    t0: int                   # first token of the rank's slice (global index)
    t1: int                   # one past its last token
    seqs: tuple               # global indices of the sequences with tokens in the slice (or empty, starting in it)
    local_cu: tuple           # cu_seqlens of those sequences, clipped to the slice and shifted to 0
    continues_in: bool        # the first local sequence started on an earlier rank
    continues_out: bool       # the last local sequence goes on past t1 on a later rank
    ends_here: tuple          # per local sequence: True if its last token (or its empty self) is in this slice


def plan_rank(cu_seqlens, t0: int, t1: int) -> RankPlan:
    """The sequences of the global ``cu_seqlens`` (host ints, [N+1]) that rank
    slice [t0, t1) computes.  An empty sequence belongs to the slice its start
    falls in (the last slice for one at the very end)."""
    cu = [int(x) for x in cu_seqlens]
    T = cu[-1]
    if not (0 <= t0 <= t1 <= T):
        raise ValueError(f"slice [{t0}, {t1}) outside the batch of {T} tokens")
    seqs, local_cu, ends = [], [0], []
    for n in range(len(cu) - 1):
        s0, s1 = cu[n], cu[n + 1]
        if s1 < s0:
            raise ValueError("cu_seqlens must be non-decreasing")
        if s1 > s0:
            mine = s0 < t1 and s1 > t0
        else:
            mine = t0 <= s0 < t1 or (s0 == T and t1 == T)
        if not mine:
            continue
        seqs.append(n)
        local_cu.append(local_cu[-1] + max(0, min(s1, t1) - max(s0, t0)))
        ends.append(s1 <= t1)
    continues_in = bool(seqs) and cu[seqs[0]] < t0
    continues_out = bool(seqs) and cu[seqs[-1] + 1] > t1
    return RankPlan(t0, t1, tuple(seqs), tuple(local_cu), continues_in, continues_out, tuple(ends))


def _prefill_carry_on_gpu():
    from . import prefill_carry
    return prefill_carry


def context_parallel_prefill(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, t0: int, t1: int,
                             init_state=None, *, group=None, prefill_fn=None):
    """This rank's part of a context-parallel prefill.

    q, k, v, a, b, z  the rank's slice of the packed streams (tokens [t0, t1)).
    cu_seqlens        the GLOBAL cu_seqlens (host ints or a CPU tensor), the
                      same on every rank.
    init_state        the global initial states [N, h_v, d_k, d_v] (or None).
    group             torch.distributed process group (default: the world);
                      ranks hold consecutive slices in rank order.
    prefill_fn        the compute, with the signature and results of
                      ``gateddeltanet_layer_gb300.prefill_carry`` (the default).

    Returns (plan, out, final_state, final_conv): the rank's output rows, and
    per local sequence its state and conv history at the end of the slice
    (final for the sequences with ``plan.ends_here``)."""
    import torch
    import torch.distributed as dist

    fn = prefill_fn or _prefill_carry_on_gpu()
    cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    plan = plan_rank(cu, t0, t1)
    if q.shape[0] != t1 - t0:
        raise ValueError(f"the slice holds {q.shape[0]} tokens, not t1 - t0 = {t1 - t0}")
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    peer = lambda r: dist.get_global_rank(group, r) if group is not None else r  # noqa: E731
    dev = q.device
    h_qk, d_k = q.shape[1:]
    h_v, d_v = v.shape[1:]
    Cc = 2 * h_qk * d_k + h_v * d_v
    n_loc = len(plan.seqs)

    carried_state = carried_conv = None
    if plan.continues_in:
        if rank == 0:
            raise ValueError("rank 0 cannot continue a sequence")
        carried_state = torch.empty((h_v, d_k, d_v), dtype=torch.float32, device=dev)
        carried_conv = torch.empty((Cc, 3), dtype=q.dtype, device=dev)
        dist.recv(carried_state, src=peer(rank - 1), group=group)
        dist.recv(carried_conv, src=peer(rank - 1), group=group)

    st = None
    if init_state is not None or carried_state is not None:
        st = torch.zeros((n_loc, h_v, d_k, d_v), dtype=torch.float32, device=dev)
        for i, n in enumerate(plan.seqs):
            if i == 0 and carried_state is not None:
                st[0].copy_(carried_state)
            elif init_state is not None:
                st[i].copy_(init_state[n])
    conv = None
    if carried_conv is not None:
        conv = torch.zeros((n_loc, Cc, 3), dtype=q.dtype, device=dev)
        conv[0].copy_(carried_conv)

    local_cu = torch.tensor(plan.local_cu, dtype=torch.int32, device=dev)
    if n_loc == 0:
        out = torch.empty((0, h_v, d_v), dtype=q.dtype, device=dev)
        fs = torch.empty((0, h_v, d_k, d_v), dtype=torch.float32, device=dev)
        fc = torch.empty((0, Cc, 3), dtype=q.dtype, device=dev)
    else:
        out, fs, fc = fn(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, local_cu, st, conv)

    if plan.continues_out:
        if rank == world - 1:
            raise ValueError("the last rank cannot hand a sequence on")
        dist.send(fs[-1].contiguous(), dst=peer(rank + 1), group=group)
        dist.send(fc[-1].contiguous(), dst=peer(rank + 1), group=group)
    return plan, out, fs, fc
