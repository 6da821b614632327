"""Expert parallelism on the host: the expert partition and the exchange plan
(``mok_ep_first_expert`` / ``mok_ep_plan``, native host code) against brute
force, and the whole exchange on ``gloo`` ranks (world sizes 2 and 3).

In the ``gloo`` test each rank runs the package's exchange (``DistExchange``:
the count exchange, the plan, every row exchange of both passes) on host
tensors; the per-rank arithmetic that on a GPU runs in the library (packing
rows in sorted order, the experts on received rows, the combines) is done
here by the float64 oracle on that rank's data.  The ranks' results, put
together, must equal the oracle run once over all tokens and all experts --
which pins the partition, the plan, the arrival order of rows (source rank,
then the source's sorted order) and the return path."""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mixture_experts_layer_side_gb300 import _lib  # noqa: E402
from mixture_experts_layer_side_gb300.ep import ExpertPartition, make_plan  # noqa: E402


@pytest.mark.parametrize("E,G", [(8, 1), (8, 2), (7, 3), (256, 8), (384, 64), (5, 5), (1024, 7)])
def test_partition_is_contiguous_and_balanced(E, G):
    p = ExpertPartition(E, G)
    assert p.bounds[0] == 0 and p.bounds[-1] == E
    sizes = [p.count(g) for g in range(G)]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    assert sum(sizes) == E
    for e in range(E):
        g = p.owner(e)
        assert p.first(g) <= e < p.first(g + 1)


def test_partition_rejects_bad_sizes():
    assert _lib.mok_ep_first_expert(4, 5, 0) == -1   # more ranks than experts
    assert _lib.mok_ep_first_expert(4, 0, 0) == -1
    assert _lib.mok_ep_first_expert(4, 2, 3) == -1
    with pytest.raises(ValueError):
        ExpertPartition(3, 4)


def brute_plan(part, rank, all_counts):
    """Rows sent, rows received and the receiver's arrival-order experts,
    written out row by row from every rank's per-expert counts."""
    G = part.G
    send = [int(sum(all_counts[rank][e] for e in range(part.first(g), part.first(g + 1)))) for g in range(G)]
    arrivals = []
    for src in range(G):
        # the source's rows in its sorted order, keeping those for this rank
        for e in range(part.E):
            for _ in range(all_counts[src][e]):
                if part.owner(e) == rank:
                    arrivals.append((src, e - part.first(rank)))
    recv = [sum(1 for s, _ in arrivals if s == src) for src in range(G)]
    return send, recv, [e for _, e in arrivals]


@pytest.mark.parametrize("E,G,seed", [(8, 2, 0), (7, 3, 1), (24, 4, 2), (5, 5, 3), (9, 1, 4)])
def test_plan_matches_brute_force(E, G, seed):
    rng = np.random.default_rng(seed)
    part = ExpertPartition(E, G)
    counts = rng.integers(0, 6, size=(G, E)).astype(np.int32)
    counts[0, :] = 0  # a rank that routes nothing
    for rank in range(G):
        El = part.count(rank)
        recv_counts = counts[:, part.first(rank):part.first(rank) + El]
        plan = make_plan(part, rank, counts[rank], recv_counts)
        send, recv, experts = brute_plan(part, rank, counts)
        assert plan.send_rows == send
        assert plan.recv_rows == recv
        assert plan.recv_expert.tolist() == experts
        assert plan.n_recv == len(experts)


def test_plan_capacity_and_bad_counts():
    part = ExpertPartition(4, 2)
    counts = np.array([3, 1, 2, 2], dtype=np.int32)
    recv = np.array([[3, 1], [5, 0]], dtype=np.int32)
    with pytest.raises(_lib.MokError) as e:
        make_plan(part, 0, counts, recv, recv_capacity=8)
    assert e.value.status == 2  # MOK_ERR_UNSUPPORTED: more rows than the receiver holds
    assert make_plan(part, 0, counts, recv, recv_capacity=9).n_recv == 9
    with pytest.raises(_lib.MokError) as e:
        make_plan(part, 0, counts, np.array([[3, -1], [5, 0]], dtype=np.int32))
    assert e.value.status == 1  # MOK_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# the exchange on gloo ranks
# ---------------------------------------------------------------------------

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def global_inputs(G, T, H, I, E, k, seed):
    rng = np.random.default_rng(seed)
    Tg = G * T
    x = rng.standard_normal((Tg, H))
    W1 = rng.standard_normal((E, H, I)) * 0.3
    W3 = rng.standard_normal((E, H, I)) * 0.3
    W2 = rng.standard_normal((E, I, H)) * 0.3
    # skewed routing: most rows to the experts of the last rank, and rank 0's
    # tokens avoid the first expert entirely
    p = np.linspace(1.0, 4.0, E)
    p = p / p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(Tg)])
    idx[:T][idx[:T] == 0] = E - 1 if k == 1 else idx[:T][idx[:T] == 0]
    s = rng.random((Tg, k)) + 0.1
    dout = rng.standard_normal((Tg, H))
    return x, idx, s, W1, W3, W2, dout


def _rank_main(rank, G, port, out_dir, dims, seed):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from mixture_experts_layer_side_gb300.ep import DistExchange, ExpertPartition, make_plan
    from oracle import moe

    T, H, I, E, k = dims
    dist.init_process_group("gloo", rank=rank, world_size=G)
    x, idx, s, W1, W3, W2, dout = global_inputs(G, T, H, I, E, k, seed)
    sl = slice(rank * T, (rank + 1) * T)
    x, idx, s, dout = x[sl], idx[sl], s[sl], dout[sl]
    part = ExpertPartition(E, G)
    e0, El = part.first(rank), part.count(rank)
    W1, W3, W2 = W1[e0:e0 + El], W3[e0:e0 + El], W2[e0:e0 + El]
    R, cap = T * k, G * T * k
    ex = DistExchange()

    # source: the schedule over all experts, rows packed in its sorted order
    sched = moe.build_schedule(idx, E)
    perm, inv = sched["perm"], sched["inv_perm"]
    counts = torch.from_numpy(sched["counts"].astype(np.int32))
    recv_counts = ex.counts(part, rank, counts)
    plan = make_plan(part, rank, counts.numpy(), recv_counts, cap)
    n = plan.n_recv
    f64 = torch.float64

    # forward: dispatch, the experts on received rows (k = 1, score 1), return, combine
    x_recv = ex.rows(torch.from_numpy(x[perm // k]), plan.send_rows, plan.recv_rows, torch.empty((cap, H), dtype=f64))
    y_recv = np.zeros((0, H))
    if n:
        y_recv, _ = moe.forward(x_recv.numpy(), plan.recv_expert[:, None], np.ones((n, 1)), W1, W3, W2)
    ys = ex.rows(torch.from_numpy(np.ascontiguousarray(y_recv)), plan.recv_rows, plan.send_rows,
                 torch.empty((R, H), dtype=f64)).numpy()
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            out[t] += s[t, j] * ys[inv[t * k + j]]

    # backward: reverse combine (dout rows and scores out), the experts' backward,
    # reverse dispatch (dX rows and score gradients back)
    s_flat = s.reshape(-1)
    dout_recv = ex.rows(torch.from_numpy(dout[perm // k]), plan.send_rows, plan.recv_rows,
                        torch.empty((cap, H), dtype=f64)).numpy()
    s_recv = ex.rows(torch.from_numpy(s_flat[perm]), plan.send_rows, plan.recv_rows,
                     torch.empty(cap, dtype=f64)).numpy()
    dx_recv, ds_recv = np.zeros((n, H)), np.zeros(n)
    dW1, dW3, dW2 = np.zeros((El, H, I)), np.zeros((El, H, I)), np.zeros((El, I, H))
    if n:
        dx_recv, dW1, dW3, dW2, ds_r = moe.backward(x_recv.numpy(), plan.recv_expert[:, None], s_recv[:, None],
                                                    W1, W3, W2, dout_recv)
        ds_recv = ds_r.reshape(-1)
    dxs = ex.rows(torch.from_numpy(np.ascontiguousarray(dx_recv)), plan.recv_rows, plan.send_rows,
                  torch.empty((R, H), dtype=f64)).numpy()
    dss = ex.rows(torch.from_numpy(np.ascontiguousarray(ds_recv)), plan.recv_rows, plan.send_rows,
                  torch.empty(R, dtype=f64)).numpy()
    dX = np.zeros((T, H))
    ds = np.zeros(R)
    for f in range(R):
        dX[f // k] += dxs[inv[f]]
        ds[f] = dss[inv[f]]
    dist.destroy_process_group()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), out=out, dX=dX, ds=ds.reshape(T, k), dW1=dW1, dW3=dW3,
             dW2=dW2, n_recv=n, recv_rows=np.array(plan.recv_rows))


@pytest.mark.parametrize("G,dims", [(2, (12, 16, 8, 6, 2)), (3, (10, 16, 8, 7, 3))])
def test_gloo_ranks_match_the_single_process_oracle(tmp_path, G, dims):
    from oracle import moe
    seed = 40 + G
    port = _free_port()
    mp.start_processes(_rank_main, args=(G, port, str(tmp_path), dims, seed), nprocs=G, join=True,
                       start_method="spawn")
    T, H, I, E, k = dims
    x, idx, s, W1, W3, W2, dout = global_inputs(G, T, H, I, E, k, seed)
    ref_out, _ = moe.forward(x, idx, s, W1, W3, W2)
    dX, dW1, dW3, dW2, ds = moe.backward(x, idx, s, W1, W3, W2, dout)
    res = [np.load(os.path.join(tmp_path, f"rank{r}.npz")) for r in range(G)]
    # the routing is skewed: the ranks receive different numbers of rows
    assert len({int(r["n_recv"]) for r in res}) > 1

    def close(got, ref, name):
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * float(np.abs(ref).max()), err_msg=name)

    close(np.concatenate([r["out"] for r in res]), ref_out, "out")
    close(np.concatenate([r["dX"] for r in res]), dX, "dX")
    close(np.concatenate([r["ds"] for r in res]), ds, "ds")
    close(np.concatenate([r["dW1"] for r in res]), dW1, "dW1")
    close(np.concatenate([r["dW3"] for r in res]), dW3, "dW3")
    close(np.concatenate([r["dW2"] for r in res]), dW2, "dW2")
