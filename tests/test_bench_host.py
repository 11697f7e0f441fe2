"""Host logic of bench.py that needs no GPU: the max-over-ranks timing
reduction and the barrier, on world_size 2 over gloo; the roofline byte
accounting."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import synthetic


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    m = bench.reduce_max(1.5 + rank, world, "cpu")
    q.put((rank, m))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.0, 1, "cpu") == 3.0


def test_algorithmic_bytes():
    wl = synthetic.WORKLOADS["vla_action_expert"]
    b, f = bench.kernel_bytes_flops(wl, wl.M, 1)
    assert b == 2 * 4096 * 1024 + 50 * 1024 + 50 * 4096 and f == 2 * 50 * 8192 * 1024
    assert bench.layer_algorithmic_bytes(wl, wl.M) == 3 * 1024 * 4096 + 4 * 50 * 1024


def test_nvfp4_layer_bytes():
    wl = synthetic.WORKLOADS["llm_decode"]
    b, f = bench.fp4_layer_bytes_flops(wl, wl.M)
    # 5120 x 17408 weights x 3: 0.5 B of code + 1/16 B of scale each; residual in and out in BF16
    assert b == 3 * 5120 * 17408 * 9 // 16 + 4 * 1 * 5120
    assert f == 6.0 * 5120 * 17408


def test_nvfp4_kernel_bytes_add_up_to_the_layer():
    """The NVFP4 launches' algorithmic bytes: the two GEMMs carry all the
    weight codes and scales and the residual stream; without the activations
    passed between them (A written by one, read by the other; X read from the
    norm) they are the layer's bytes.  The norm reads the residual and its
    weight and writes X."""
    for name in ("llm_decode", "vla_action_expert", "long_prefill"):
        wl = synthetic.WORKLOADS[name]
        M, d, ff = wl.M, wl.d, wl.ff
        n, g, w = (bench.fp4_kernel_bytes_flops(wl, M, s) for s in range(3))
        x = M * d // 2 + M * d // 16     # X codes + scales: written by the norm, read by the gate/up GEMM
        a = M * ff // 2 + M * ff // 16   # A codes + scales: written by the gate/up GEMM, read by the down GEMM
        layer_b, layer_f = bench.fp4_layer_bytes_flops(wl, M)
        assert g[0] + w[0] - x - 2 * a == layer_b
        assert n[0] == 2 * M * d + 2 * d + x
        assert n[1] + g[1] + w[1] == layer_f
    # the decode gate/up figure the profile summary divides by
    wl = synthetic.WORKLOADS["llm_decode"]
    assert bench.fp4_kernel_bytes_flops(wl, 1, 1)[0] == 100282752
    assert bench.fp4_kernel_bytes_flops(wl, 1, 2)[0] == 50165312


def test_l2_note_states_the_flush(monkeypatch):
    assert bench.l2_note().startswith("flushed")
    monkeypatch.setattr(bench, "WARM_L2", True)
    assert bench.l2_note().startswith("warm")
    assert bench.config_of(synthetic.WORKLOADS["tiny"])["l2"].startswith("warm")
