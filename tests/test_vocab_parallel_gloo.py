"""The vocabulary-parallel exchange on CPU ranks (gloo): two, three and eight.

Each rank holds half of the vocabulary, computes its shard's softmax statistics with
the oracle, exchanges them with the package's exchange_stats (an all-gather), merges
them, and sums its shard's dhidden term with reduce_dhidden (an all-reduce).  The
results must equal the whole-vocabulary oracle: this covers the collective steps of
the sharded path without a GPU.
"""
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


def _worker(rank, world, port, reduction, cap):
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from linear_cross_entropy_forward_gb300.vocab_parallel import exchange_stats, reduce_dhidden
    from oracle import flce_oracle as orc
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        rng = np.random.default_rng(7)
        N, H, V = 19, 11, 83
        hidden = rng.standard_normal((N, H))
        weight = rng.standard_normal((H, V)) * 0.9
        labels = rng.integers(0, V, N)
        labels[[2, 9]] = orc.IGNORE_INDEX
        g_loss = rng.standard_normal(N) if reduction == "none" else np.array([0.8])
        g_ent = rng.standard_normal(N) if reduction == "none" else np.array([-0.6])
        cuts = np.linspace(0, V, world + 1).astype(int)
        a, b = int(cuts[rank]), int(cuts[rank + 1])
        local = torch.from_numpy(orc.shard_stats(hidden, weight[:, a:b], labels, a, cap))
        gathered = exchange_stats(local)
        assert gathered.shape == (world, 4, N)
        comb = orc.combine_shards(gathered.numpy(), labels, reduction, zloss_coef=0.01,
                                  v_total=V)
        whole = orc.forward(hidden, weight, labels, reduction, zloss_coef=0.01, softcap=cap)
        np.testing.assert_allclose(comb["loss"], whole["loss"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(comb["entropy"], whole["entropy"], rtol=1e-12, atol=1e-12)
        dh_part, dw_part = orc.backward(hidden, weight[:, a:b], labels, comb["lse"], comb["ez"],
                                        g_loss, g_ent, reduction, zloss_coef=0.01, softcap=cap,
                                        v_offset=a, v_total=V)
        dh = reduce_dhidden(torch.from_numpy(dh_part)).numpy()
        dh_w, dw_w = orc.backward(hidden, weight, labels, whole["lse"], whole["ez"], g_loss,
                                  g_ent, reduction, zloss_coef=0.01, softcap=cap)
        np.testing.assert_allclose(dh, dh_w, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dw_part, dw_w[:, a:b], rtol=1e-11, atol=1e-13)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("reduction,cap", [("mean", 0.0), ("none", 2.0), ("sum", 0.0)])
def test_two_rank_vocab_parallel_exchange(reduction, cap):
    mp.spawn(_worker, args=(2, _free_port(), reduction, cap), nprocs=2, join=True)


def test_three_rank_vocab_parallel_exchange():
    mp.spawn(_worker, args=(3, _free_port(), "mean", 1.5), nprocs=3, join=True)


def test_eight_rank_vocab_parallel_exchange():
    """Eight shards of 10-11 columns each: the all-gather of the statistics, the merge and
    the all-reduce of the dhidden terms against the whole-vocabulary oracle."""
    mp.spawn(_worker, args=(8, _free_port(), "none", 2.0), nprocs=8, join=True)


def _worker_peer_leaves(rank, world, port, flag_path):
    """Rank 1 leaves before the exchange (between steps, nothing in flight); rank 0's
    exchange must end with an error within the process group's timeout, not hang."""
    import datetime
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from linear_cross_entropy_forward_gb300.vocab_parallel import exchange_stats
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(0)  # the rank is gone: no destroy, no further collective
    try:
        exchange_stats(torch.zeros(4, 8, dtype=torch.float64))
    except Exception as e:  # gloo reports the lost peer (or the timeout) as an error
        with open(flag_path, "w") as f:
            f.write(type(e).__name__)
    finally:
        os._exit(0)


def test_exchange_reports_a_rank_that_left(tmp_path):
    flag = tmp_path / "detected"
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker_peer_leaves, args=(r, 2, port, str(flag)))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=60)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a rank hung instead of reporting the lost peer"
    assert flag.exists(), "rank 0's exchange did not raise"


def _worker_bf16_sum(rank, world, port, path):
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from linear_cross_entropy_forward_gb300.vocab_parallel import reduce_dhidden
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        g = torch.Generator().manual_seed(100 + rank)
        part = torch.randn(33, 17, generator=g).to(torch.bfloat16)
        out = reduce_dhidden(part)
        assert out.dtype == torch.bfloat16 and out.shape == part.shape
        torch.save((part, out), f"{path}.{rank}")
    finally:
        dist.destroy_process_group()


def test_reduce_dhidden_sums_bf16_terms_in_fp32(tmp_path):
    """dhidden terms arrive in bf16; they are summed in fp32 across the ranks and rounded
    once, so every rank gets the same, once-rounded sum."""
    path = str(tmp_path / "r")
    mp.spawn(_worker_bf16_sum, args=(2, _free_port(), path), nprocs=2, join=True)
    (a, out0), (b, out1) = torch.load(f"{path}.0"), torch.load(f"{path}.1")
    want = (a.float() + b.float()).to(torch.bfloat16)
    assert torch.equal(out0, want) and torch.equal(out1, want)
