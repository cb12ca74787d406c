"""Expert-parallel dispatch and combine across CPU ranks (gloo, world sizes 2 and 4).

Every rank holds a slice of the tokens (one rank holds none) and E/G of the
experts; a router bias keeps the last rank's experts unselected, so that rank
receives no rows.  The routed part of the layer computed through plan -> dispatch
-> local experts -> return -> combine must equal the single-process oracle: the
routing bit for bit and y bit for bit in fp64 (the combine adds the same products
in the same order as the oracle does).  The local experts are evaluated by the
oracle here (one forced expert per row, weight exactly 1), so these tests check
the bookkeeping and the exchange; a GPU test runs the library's local experts.
"""
import dataclasses
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer(family, world):
    import moe_inputs as mi
    if family == "qwen":
        spec = mi.small_spec("qwen", 64, 8, 2, 32, 0, 21)
    else:
        spec = mi.small_spec("gptoss", 64, 8, 2, 64, 0, 21)
    lay = mi.make_layer(spec)
    # the last rank's experts never win: that rank receives no rows
    epr = spec.n_experts // world
    b = np.zeros(spec.n_experts)
    b[spec.n_experts - epr:] = -30.0
    lay.router_b = mi.f64_to_bf16(b)
    return spec, lay


def _splits(world, T):
    return {2: [13, 8], 4: [9, 0, 5, 7]}[world] if T == 21 else None


def _oracle_local_experts(g, lay, lo, hi):
    """local_experts(rows, local_ids) evaluated by the oracle: a layer of experts
    [lo, hi) with zero router weights, one forced expert per row, so that the routing
    weight is exactly 1 and y is that expert's output."""
    import oracle
    kw = {}
    for name in ("gate", "up", "down", "gate_up", "gu_blocks", "gu_scales", "gu_bias", "dn_blocks",
                 "dn_scales", "dn_bias"):
        a = getattr(lay, name)
        kw[name] = None if a is None else np.ascontiguousarray(a[lo:hi])
    local = dataclasses.replace(lay, router_w=np.zeros((hi - lo, g.d_model), np.uint16), router_b=None,
                                sh_gate=None, sh_up=None, sh_down=None, sh_gate_inp=None, **kw)
    gl = dataclasses.replace(g, n_experts=hi - lo, top_k=1, shared_ff=0)

    def run(rows, local_ids):
        R = rows.shape[0]
        if R == 0:
            return torch.empty((0, g.d_model), dtype=torch.float64)
        x = rows.numpy().astype(np.uint16)
        res = oracle.forward(gl, local, x=x, forced_ids=local_ids.numpy().reshape(R, 1))
        assert np.all(res.w == 1.0)
        return torch.from_numpy(res.y)

    return run


def _rank(rank, world, port, family, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from sparse_moe_ffn_route_gb300 import expert_parallel as ep
        spec, lay = _layer(family, world)
        g = oracle.gating_for(spec)
        sp = _splits(world, spec.tokens)
        first = sum(sp[:rank])
        mine = np.arange(first, first + sp[rank], dtype=np.int32)
        # this rank's routing (data-parallel router)
        r = oracle.route(g, lay, tokens=mine)
        ids = torch.from_numpy(r.ids.copy())
        w = torch.from_numpy(r.w.copy())
        # bf16 bit patterns travel as int32 (gloo has no 16-bit integer type)
        x = torch.from_numpy(lay.x[mine].astype(np.int32))
        epr = spec.n_experts // world
        local = _oracle_local_experts(g, lay, rank * epr, (rank + 1) * epr)
        plan = ep.dispatch_plan(ids, spec.n_experts)
        rows = ep.dispatch(x, plan)
        # the rows that arrived are the token rows of the slots that chose this rank's experts
        Y = local(rows, plan.recv_local_ids)
        y = ep.combine(ep.gather_back(Y, plan), w)
        # round trip of the slot indices themselves: every slot comes back to its place
        slot_ids = torch.arange(len(mine) * spec.top_k, dtype=torch.float64).view(-1, 1)
        sent = slot_ids.index_select(0, plan.send_order)
        there = torch.empty((plan.rows_received, 1), dtype=torch.float64)
        torch.distributed.all_to_all_single(there, sent, plan.recv_counts, plan.send_counts)
        back = ep.gather_back(there, plan)
        ref = oracle.forward(g, lay)       # the single-process layer, every token
        q.put({"rank": rank, "tokens": len(mine), "received": plan.rows_received,
               "sent": plan.send_counts, "roundtrip": bool(torch.equal(back, slot_ids)),
               "ids_equal": bool(np.array_equal(r.ids, ref.ids[mine])),
               "y_equal": bool(np.array_equal(y.numpy(), ref.y[mine])),
               "max_diff": float(np.max(np.abs(y.numpy() - ref.y[mine]))) if len(mine) else 0.0,
               "local_ids_ok": bool(plan.recv_local_ids.numel() == 0 or
                                    (int(plan.recv_local_ids.min()) >= 0 and
                                     int(plan.recv_local_ids.max()) < epr))})
    except Exception as e:   # report instead of hanging the other ranks' queue reads
        q.put({"rank": rank, "error": repr(e)})
        raise
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("family", ["qwen", "gptoss"])
def test_expert_parallel_matches_single_process_oracle(world, family):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, family, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(120)
    for d in res:
        assert "error" not in d, d
    for p in procs:
        assert p.exitcode == 0
    spec_T, k = 21, 2
    assert sum(d["tokens"] for d in res) == spec_T
    assert sum(d["received"] for d in res) == spec_T * k          # every slot went somewhere once
    assert res[-1]["received"] == 0                                 # the biased-out rank got nothing
    assert all(d["sent"][-1] == 0 for d in res)
    if world == 4:
        assert res[1]["tokens"] == 0 and sum(res[1]["sent"]) == 0  # a rank without tokens
    for d in res:
        assert d["roundtrip"] and d["ids_equal"] and d["local_ids_ok"], d
        assert d["y_equal"], d


def _forward_rank(rank, world, port, q):
    """ep.forward end to end on one rank, with stand-in experts: expert e maps a row r
    to (e + 1) * r, so the result is known in closed form."""
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sparse_moe_ffn_route_gb300 import expert_parallel as ep
        E, k, d = 8, 3, 5
        T = [4, 0, 7, 2][rank] if world == 4 else [6, 3][rank]
        g = torch.Generator().manual_seed(100 + rank)
        x = torch.randn(T, d, generator=g, dtype=torch.float64)
        ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32) \
            if T else torch.empty((0, k), dtype=torch.int32)
        w = torch.rand(T, k, generator=g, dtype=torch.float64)
        epr = E // world

        def local(rows, local_ids):
            return rows * (local_ids.to(torch.float64) + rank * epr + 1.0).unsqueeze(1)

        y = ep.forward(x, ids, w, E, local)
        want = torch.zeros((T, d), dtype=torch.float64)
        for j in range(k):
            want = want + w[:, j:j + 1] * (x * (ids[:, j:j + 1].to(torch.float64) + 1.0))
        q.put({"rank": rank, "ok": bool(torch.equal(y, want)), "T": T})
    except Exception as e:
        q.put({"rank": rank, "error": repr(e)})
        raise
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_forward_end_to_end_with_stand_in_experts(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_forward_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(120)
    for d in res:
        assert "error" not in d and d["ok"], d


def test_owner_blocks_and_uneven_split_rejected():
    from sparse_moe_ffn_route_gb300 import expert_parallel as ep
    ids = torch.tensor([[0, 7], [3, 4]], dtype=torch.int32)
    assert ep.owner_of(ids, 8, 4).tolist() == [[0, 3], [1, 2]]
    assert ep.owner_of(ids, 8, 2).tolist() == [[0, 1], [0, 1]]
    with pytest.raises(ValueError):
        ep.owner_of(ids, 8, 3)


def test_combine_adds_slots_in_order():
    from sparse_moe_ffn_route_gb300 import expert_parallel as ep
    Y = torch.tensor([[1.0, 2.0], [10.0, 20.0], [3.0, 4.0], [30.0, 40.0]], dtype=torch.float64)
    w = torch.tensor([[0.25, 0.75], [0.5, 0.5]], dtype=torch.float64)
    y = ep.combine(Y, w)
    assert y.tolist() == [[0.25 * 1 + 0.75 * 10, 0.25 * 2 + 0.75 * 20], [0.5 * 3 + 0.5 * 30, 0.5 * 4 + 0.5 * 40]]
