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


HP = dict(lr=1e-2, b1=0.9, b2=0.999, eps=1e-8, wd=0.01)
STEPS = 3


def _bf16_bits(x64):
    import oracle
    return np.vectorize(oracle.bf16_round_d, otypes=[np.uint16])(x64)


def _train(rank, world, reduce_fn):
    """A few steps of the data-parallel loop on this rank's token shard: fp64 master adapters,
    their bf16 copies feed the layer, the shard's dA and dB are summed over ranks, and every rank
    applies the same AdamW step to its own replica."""
    import oracle
    inp = _layer()
    M = inp.X.shape[0]
    lo, hi = rank * M // world, (rank + 1) * M // world
    A, B = oracle.bf16_to_f64(inp.A), oracle.bf16_to_f64(inp.B)
    st = {k: np.zeros(A.size if k[0] == "A" else B.size) for k in ("Am", "Av", "Bm", "Bv")}
    for t in range(1, STEPS + 1):
        Ab, Bb = _bf16_bits(A), _bf16_bits(B)
        dA, dB = oracle.layer_adapter_grads(inp.X[lo:hi], Ab, Bb, inp.G[lo:hi], inp.alpha)
        dA, dB = reduce_fn(dA), reduce_fn(dB)
        a, st["Am"], st["Av"] = oracle.adamw_step(A, dA, st["Am"], st["Av"], HP["lr"], HP["b1"], HP["b2"], HP["eps"],
                                                  HP["wd"], t)
        b, st["Bm"], st["Bv"] = oracle.adamw_step(B, dB, st["Bm"], st["Bv"], HP["lr"], HP["b1"], HP["b2"], HP["eps"],
                                                  HP["wd"], t)
        A, B = a.reshape(A.shape), b.reshape(B.shape)
    return dict(A=A, B=B, **st)


def _train_rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def all_reduce(x):
        t = torch.from_numpy(np.ascontiguousarray(x))
        dist.all_reduce(t)
        return t.numpy()

    np.savez(os.path.join(out_dir, f"train{rank}.npz"), **_train(rank, world, all_reduce))
    dist.destroy_process_group()


def test_replicas_stay_identical_through_adamw_steps(orc, tmp_path):
    """Three data-parallel steps (gradient all-reduce, then AdamW on each replica): the two
    replicas' adapters and moments are equal bit for bit, and equal the single-process full-batch
    loop up to the summation order of the gradients."""
    world = 2
    mp.start_processes(_train_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r0, r1 = (np.load(tmp_path / f"train{k}.npz") for k in range(world))
    ref = _train(0, 1, lambda x: x)
    inp = _layer()
    assert not np.array_equal(r0["A"], orc.bf16_to_f64(inp.A))  # the adapters did move
    for k in ("A", "B", "Am", "Av", "Bm", "Bv"):
        np.testing.assert_array_equal(r0[k], r1[k], err_msg=k)
        np.testing.assert_allclose(r0[k], ref[k], rtol=1e-9, atol=1e-15, err_msg=k)
