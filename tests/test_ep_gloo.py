"""Expert parallelism, simulated on CPU ranks with the oracle (no GPU path: one GPU per run).

[MoE] "The traceable trick: compute all experts, mask to top-8" shards the experts over 8 ranks
(rank r owns experts 16 r .. 16 r + 15: gate_up column-parallel, down row-parallel) and adds the
ranks' partial expert outputs with an all-reduce. These tests pin that decomposition of the block:

* A rank's partial is the block's expert branch with the weights of the other ranks' experts set
  to zero (per_expert_scale masked). The top-8 choice is taken on the logits, so it is the same on
  every rank and equal to the unsharded one.
* The partials summed over the ranks give the expert branch, and the block output follows from that
  sum through the post norms. The exchange has to come before post_feedforward_layernorm_2: the
  same norms applied per rank and summed afterwards give a different block.
* With world size 2 on gloo, an all-reduce of the two ranks' partials reproduces the output.
* bench.py's expert-parallel step (its expert ranges, the all-reduce of the partials and the
  broadcast of rank 0's shared-MLP output, then the finishing arithmetic), run by two gloo ranks
  with oracle shards, reproduces the output on both ranks.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
from mixture_experts_ffn_router_gb300 import synth
from tests import tiny

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _shard_weights(w: dict, experts: range) -> dict:
    """The weights one rank runs: per_expert_scale zero outside its experts (the router inputs,
    and so the top-8 choice, are untouched)."""
    ws = dict(w)
    pes = np.zeros_like(np.asarray(w["per_expert_scale"], dtype=np.float32))
    pes[list(experts)] = np.asarray(w["per_expert_scale"], dtype=np.float32)[list(experts)]
    ws["per_expert_scale"] = pes
    return ws


def _x_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _norm_rows(v, wn, eps):
    return np.stack([oracle.rmsnorm(v[t], wn, eps) for t in range(v.shape[0])])


def _block_from_normed(moe_n, dense, x_bits, w, eps):
    """Block output from the normalised expert branch and the shared-MLP branch ([MoE] "The
    architecture": both branches normalised, summed, normalised, residual added, times
    layer_scalar)."""
    y = _norm_rows(_norm_rows(dense, w["post_ff_ln_1"], eps) + moe_n, w["post_ff_ln"], eps)
    return (_x_f64(x_bits) + y) * float(np.float32(w["layer_scalar"]))  # an fp32 field of the weights


def _block_from_branches(moe, dense, x_bits, w, eps):
    return _block_from_normed(_norm_rows(moe, w["post_ff_ln_2"], eps), dense, x_bits, w, eps)


def _ranks(E: int, n: int):
    per = E // n
    return [range(r * per, (r + 1) * per) for r in range(n)]


@pytest.mark.parametrize("shape,T,n_ranks,seed", [(tiny.SMALL, 12, 8, 31), (tiny.SMALL, 5, 2, 32)])
def test_expert_shards_sum_to_the_block(shape, T, n_ranks, seed):
    d = tiny.dims_of(shape, full_layer=True)
    x, w = tiny.case(shape, T, seed, weight_std=0.2)
    want = ("out", "moe", "dense", "topk_idx")
    full = oracle.forward(d, x, w, want=want)
    parts = []
    for experts in _ranks(shape["n_experts"], n_ranks):
        r = oracle.forward(d, x, _shard_weights(w, experts), want=want)
        np.testing.assert_array_equal(r["topk_idx"], full["topk_idx"])  # the choice does not move
        np.testing.assert_array_equal(r["dense"], full["dense"])          # the shared MLP is replicated
        # a token none of whose 8 experts this rank owns gets an exact zero from it
        owns = np.isin(full["topk_idx"], list(experts)).any(axis=1)
        assert np.all(r["moe"][~owns] == 0.0)
        parts.append(r)
    moe_sum = np.sum([p["moe"] for p in parts], axis=0)
    np.testing.assert_allclose(moe_sum, full["moe"], rtol=1e-12, atol=1e-14)
    out = _block_from_branches(moe_sum, full["dense"], x, w, d["eps"])
    np.testing.assert_allclose(out, full["out"], rtol=1e-12, atol=1e-12)
    # Normalising each rank's partial with post_feedforward_layernorm_2 before the exchange gives a
    # different block: the all-reduce has to come first.
    moe_n_wrong = np.sum([_norm_rows(p["moe"], w["post_ff_ln_2"], d["eps"]) for p in parts], axis=0)
    wrong = _block_from_normed(moe_n_wrong, full["dense"], x, w, d["eps"])
    assert np.max(np.abs(wrong - full["out"])) > 1e-2


def test_expert_shards_at_the_model_shapes():
    # Hidden 2816, 128 experts, top-8, 8 ranks of 16 experts each, as the pages shard them.
    shape = synth.GEMMA
    d = oracle.gemma_dims(True)
    T = 3
    x = synth.bf16_bits(synth.make_x(T, seed=41))
    w = synth.host_arrays(synth.make_weights(seed=41, full_layer=True))
    want = ("out", "moe", "dense", "topk_idx")
    full = oracle.forward(d, x, w, want=want)
    moe_sum = np.zeros_like(full["moe"])
    for experts in _ranks(shape["n_experts"], 8):
        r = oracle.forward(d, x, _shard_weights(w, experts), want=want)
        np.testing.assert_array_equal(r["topk_idx"], full["topk_idx"])
        moe_sum += r["moe"]
    np.testing.assert_allclose(moe_sum, full["moe"], rtol=1e-12, atol=1e-14)
    out = _block_from_branches(moe_sum, full["dense"], x, w, d["eps"])
    np.testing.assert_allclose(out, full["out"], rtol=1e-12, atol=1e-12)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from tests import tiny as tn
    import oracle as orc
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = tn.SMALL
    d = tn.dims_of(shape, full_layer=True)
    x, w = tn.case(shape, 9, 57, weight_std=0.2)  # every rank draws the same seeded layer and batch
    experts = _ranks(shape["n_experts"], world)[rank]
    part = orc.forward(d, x, _shard_weights(w, experts), want=("moe", "dense"))
    moe = torch.from_numpy(part["moe"].copy())
    dist.all_reduce(moe, op=dist.ReduceOp.SUM)  # the exchange step of the row-parallel down
    out = _block_from_branches(moe.numpy(), part["dense"], x, w, d["eps"])
    q.put((rank, out))
    dist.destroy_process_group()


def test_expert_parallel_all_reduce_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    shape = tiny.SMALL
    d = tiny.dims_of(shape, full_layer=True)
    x, w = tiny.case(shape, 9, 57, weight_std=0.2)
    full = oracle.forward(d, x, w, want=("out",))
    for r in (0, 1):
        np.testing.assert_allclose(res[r], full["out"], rtol=1e-12, atol=1e-12)


def _bench_rank_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    from tests import tiny as tn
    import oracle as orc
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = tn.SMALL
    d = tn.dims_of(shape, full_layer=True)
    x, w = tn.case(shape, 7, 61, weight_std=0.2)

    def shard(b, e, with_dense):
        r = orc.forward(d, x, _shard_weights(w, range(b, e)), want=("moe", "dense"))
        part = torch.from_numpy(r["moe"].copy())
        dense = torch.from_numpy(r["dense"].copy()) if with_dense else torch.zeros_like(part)
        return part, dense

    out = bench.ep_rank_step(rank, world, shard, lambda p, dd: bench.ep_exchange(p, dd, world, dist),
                             lambda p, dd: _block_from_branches(p.numpy(), dd.numpy(), x, w, d["eps"]),
                             n_experts=shape["n_experts"])
    q.put((rank, out))
    dist.destroy_process_group()


def test_bench_expert_parallel_step_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bench_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    shape = tiny.SMALL
    d = tiny.dims_of(shape, full_layer=True)
    x, w = tiny.case(shape, 7, 61, weight_std=0.2)
    full = oracle.forward(d, x, w, want=("out",))
    for r in (0, 1):
        np.testing.assert_allclose(res[r], full["out"], rtol=1e-12, atol=1e-12)
