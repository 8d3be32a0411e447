"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2): each rank
reports its own timed region, the job takes the maximum, and only rank 0
prints.  By default ranks are independent replicas; with --dp-allreduce the
weight gradients are summed over the ranks after every backward, through the
same function tested here on CPU tensors."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier()
    got = bench.max_over_ranks(10.0 + rank * 5.0)
    ws, r, lr = bench.dist_env()
    dist.destroy_process_group()
    with open(out, "w") as f:
        json.dump({"max": got, "ws": ws, "rank": r, "local": lr}, f)


def test_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    outs = [str(tmp_path / ("r%d.json" % r)) for r in range(2)]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, port, outs[r])) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(o)) for o in outs]
    assert all(r["max"] == 15.0 for r in res)
    assert sorted(r["rank"] for r in res) == [0, 1] and all(r["ws"] == 2 for r in res)


def _grad_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank's fp32 gradient increments of its own tokens (as the backward
    # leaves them), two buffers of the shapes dW13 [E, 2I, d] and dW2 [E, d, I]
    g = torch.Generator().manual_seed(100 + rank)
    dw13 = torch.randn(3, 8, 16, generator=g)
    dw2 = torch.randn(3, 16, 4, generator=g)
    mine = (dw13.clone(), dw2.clone())
    bench.allreduce_grads((dw13, dw2))
    dist.destroy_process_group()
    torch.save({"mine": mine, "sum": (dw13, dw2)}, out)


def test_dp_allreduce_sums_weight_gradients_gloo(tmp_path):
    import torch
    import torch.multiprocessing as mp

    port = _free_port()
    outs = [str(tmp_path / ("g%d.pt" % r)) for r in range(2)]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_grad_worker, args=(r, 2, port, outs[r])) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [torch.load(o) for o in outs]
    for i in range(2):
        want = res[0]["mine"][i] + res[1]["mine"][i]
        assert torch.allclose(res[0]["sum"][i], want) and torch.equal(res[0]["sum"][i],
                                                                      res[1]["sum"][i])


def test_reference_arm_prints_only_on_rank0():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         env=env, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_stage_model_counts_the_method_flops():
    sys.path.insert(0, ROOT)
    import bench

    c = dict(T=8192, d=2048, I=768, E=128, k=8)
    m = bench.stage_model(c)
    R = 8192 * 8
    fwd = m["w13_swiglu"][1] + m["w2_score"][1]
    bwd = sum(m[s][1] for s in ("dgrad_w2_swiglu", "dgrad_w13", "wgrad_w2", "wgrad_w13"))
    assert fwd == 6 * R * 2048 * 768
    assert fwd + bwd == 18 * R * 2048 * 768


def test_kernel_hash_ignores_comments_only():
    """The committed DRAM counters stay tied to the kernels' code: a comment or
    layout edit keeps the hash, a code edit (also inside a string) changes it."""
    sys.path.insert(0, ROOT)
    import bench

    a = 'int f(int x) { // twice\n  return 2 * x; /* no\n overflow */ }\nconst char* s = "// kept";\n'
    b = 'int f(int x) {\n    return 2 * x;\n}\nconst char* s = "// kept";  // the same code\n'
    c = 'int f(int x) { return 3 * x; }\nconst char* s = "// kept";\n'
    d = 'int f(int x) { return 2 * x; }\nconst char* s = "// changed";\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)
    assert "kept" in bench._code_only(a)
