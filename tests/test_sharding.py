"""Data-parallel sharding of the path, checked with the oracle on CPU.

Every 16-element block is independent, so the path shards over tokens: Fprop
and Dgrad over M, Wgrad over K (its partial products sum to the full one: the
ordinary data-parallel gradient all-reduce).  The one cross-shard dependency
is the tensor amax, a scalar max all-reduce.  Two gloo ranks each quantize
their half of the tokens with the all-reduced amax and compute their partial
Wgrad; the combined results must equal the unsharded oracle: codes and scales
byte for byte, the Wgrad sum to FP64 rounding.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from fp4_gemm_nvfp4_gb300 import inputs

TOKENS, HIDDEN, OUT = 96, 128, 48


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tensors():
    x = inputs.normal(TOKENS, HIDDEN, seed=21, outlier_channels=1)
    dy = inputs.student_t(TOKENS, OUT, seed=22)
    return x, dy


def _worker(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        x, dy = _tensors()
        per = TOKENS // world
        r0, r1 = rank * per, (rank + 1) * per
        # Fprop input, row-wise over this rank's tokens, with the agreed amax
        local_amax = torch.tensor([float(oracle.amax(x[r0:r1]))], dtype=torch.float32)
        dist.all_reduce(local_amax, op=dist.ReduceOp.MAX)
        qx = oracle.quantize(x, oracle.ROWWISE, rounding=1, seed=7, rows_subset=(r0, r1),
                             amax_value=np.float32(local_amax.item()))
        # Wgrad partial: dY^T X over this rank's tokens (K = tokens), both
        # operands col-wise so that K is contiguous
        qa = oracle.quantize(dy, oracle.COLWISE)
        qb = oracle.quantize(x, oracle.COLWISE)
        k0, k1 = r0, r1
        part_a = dict(codes=qa["codes"][:, k0 // 2:k1 // 2], scales=qa["scales"][:, k0 // 16:k1 // 16], s_g=qa["s_g"])
        part_b = dict(codes=qb["codes"][:, k0 // 2:k1 // 2], scales=qb["scales"][:, k0 // 16:k1 // 16], s_g=qb["s_g"])
        y, _ = oracle.gemm_f64(part_a, part_b, with_abs=False)
        yt = torch.from_numpy(y.copy())
        dist.all_reduce(yt, op=dist.ReduceOp.SUM)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), codes=qx["codes"], scales=qx["scales"],
                 amax=np.float32(local_amax.item()), wgrad=yt.numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_token_sharding_matches_unsharded_oracle(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    x, dy = _tensors()
    full = oracle.quantize(x, oracle.ROWWISE, rounding=1, seed=7)
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    for p in parts:
        assert p["amax"] == full["amax"]
    np.testing.assert_array_equal(np.concatenate([p["codes"] for p in parts]), full["codes"])
    np.testing.assert_array_equal(np.concatenate([p["scales"] for p in parts]), full["scales"])
    y_full, _ = oracle.gemm_f64(oracle.quantize(dy, oracle.COLWISE), oracle.quantize(x, oracle.COLWISE),
                                with_abs=False)
    for p in parts:
        np.testing.assert_allclose(p["wgrad"], y_full, rtol=1e-12, atol=1e-300)
