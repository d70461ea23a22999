"""Data-parallel QLoRA layer on CPU with gloo (world size 2): tokens are sharded across ranks, the
forward and dX need no exchange, and summing each rank's dA, dB with one all-reduce gives the
full-batch adapter gradients -- the one collective of a data-parallel step.  Uses the oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer(seed=31, M=12, N=24, K=128, r=4):
    from bit_nf4_quantized_36_b300 import synth
    inp = synth.layer_inputs(seed, M, N, K, r, 8.0, b_std=0.3)
    return inp


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    inp = _layer()
    M = inp.X.shape[0]
    lo, hi = rank * M // world, (rank + 1) * M // world
    q = oracle.nf4_quantize(inp.W)
    N, K = inp.W.shape
    What = oracle.nf4_dequantize(q["packed"], q["qcode"], q["c2"], q["mu"], N, K)
    Y, _ = oracle.layer_fwd_rows(What, inp.X[lo:hi], inp.A, inp.B, inp.alpha)
    dX = oracle.layer_dx_rows(What, inp.A, inp.B, inp.G[lo:hi], inp.alpha)
    dA, dB = oracle.layer_adapter_grads(inp.X[lo:hi], inp.A, inp.B, inp.G[lo:hi], inp.alpha)
    tA, tB = torch.from_numpy(dA), torch.from_numpy(dB)
    dist.all_reduce(tA)
    dist.all_reduce(tB)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), Y=Y, dX=dX, dA=tA.numpy(), dB=tB.numpy(), lo=lo, hi=hi)
    dist.destroy_process_group()


def test_token_sharded_step_equals_full_batch(orc, tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    inp = _layer()
    N, K = inp.W.shape
    q = orc.nf4_quantize(inp.W)
    What = orc.nf4_dequantize(q["packed"], q["qcode"], q["c2"], q["mu"], N, K)
    Y, _ = orc.layer_fwd_rows(What, inp.X, inp.A, inp.B, inp.alpha)
    dX = orc.layer_dx_rows(What, inp.A, inp.B, inp.G, inp.alpha)
    dA, dB = orc.layer_adapter_grads(inp.X, inp.A, inp.B, inp.G, inp.alpha)
    for rank in range(world):
        d = np.load(tmp_path / f"rank{rank}.npz")
        lo, hi = int(d["lo"]), int(d["hi"])
        np.testing.assert_allclose(d["Y"], Y[lo:hi], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(d["dX"], dX[lo:hi], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(d["dA"], dA, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(d["dB"], dB, rtol=1e-11, atol=1e-12)
