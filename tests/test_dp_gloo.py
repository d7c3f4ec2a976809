"""World-size-2 data-parallel exchange on CPU (gloo): the summed sketch equals
the sketch of all ranks' micro-batches, and the global q(D) equals the mean
over all ranks' rows.  The per-rank values come from the oracle; what is under
test is the exchange logic of rank_gradient_sketching_gb300/dp.py, loaded by
path so that no GPU library is needed."""

import importlib.util
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_dp():
    spec = importlib.util.spec_from_file_location("_logra_dp", os.path.join(ROOT, "rank_gradient_sketching_gb300",
                                                                              "dp.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(rank):
    g = torch.Generator().manual_seed(100 + rank)
    X = (torch.randn((64, 40), generator=g)).to(torch.bfloat16).double().numpy()
    dY = (torch.randn((64, 24), generator=g) * 1e-3).to(torch.bfloat16).double().numpy()
    rows = 3 + 2 * rank  # unequal row counts per rank
    cur = (torch.randn((rows, 50), generator=g) * 2).double().numpy()
    prop = cur + 0.1 * torch.randn((rows, 50), generator=g).double().numpy()
    return X, dY, cur, prop


def _worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    from oracle import kl as okl
    from oracle import philox as oph
    from oracle import sketch as osk

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    dp = _load_dp()
    X, dY, cur, prop = _inputs(rank)
    A = oph.projection(7, 3, 8, 40)
    S = osk.sketch_accumulate(np.zeros((24, 8)), [(X, dY)], A)
    s_flat = torch.tensor(S.reshape(-1), dtype=torch.float32)
    dp.allreduce_sketch(s_flat)
    q, _ = okl.predicted_kl(cur, prop, 1.0)
    q_t = torch.tensor(q, dtype=torch.float64)
    dp.global_q(q_t, cur.shape[0])
    np.save(os.path.join(out_dir, f"S{rank}.npy"), s_flat.numpy())
    np.save(os.path.join(out_dir, f"q{rank}.npy"), np.array([q_t.item()]))
    torch.distributed.destroy_process_group()


def test_two_rank_exchange(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    from oracle import kl as okl
    from oracle import philox as oph
    from oracle import sketch as osk

    ins = [_inputs(r) for r in range(world)]
    A = oph.projection(7, 3, 8, 40)
    S_all = osk.sketch_accumulate(np.zeros((24, 8)), [(X, dY) for X, dY, _, _ in ins], A)
    q_all, _ = okl.predicted_kl(np.concatenate([c for _, _, c, _ in ins]), np.concatenate([p for _, _, _, p in ins]),
                                1.0)
    for r in range(world):
        S_r = np.load(tmp_path / f"S{r}.npy").reshape(24, 8)
        assert np.allclose(S_r, S_all, rtol=1e-5, atol=1e-9)
        assert abs(np.load(tmp_path / f"q{r}.npy")[0] - q_all) <= 1e-12 * abs(q_all)
    # both ranks hold the same sketch afterwards, so their merges agree
    assert np.array_equal(np.load(tmp_path / "S0.npy"), np.load(tmp_path / "S1.npy"))


def _payload_worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    dp = _load_dp()
    payload = None
    if rank == 0:
        g = torch.Generator().manual_seed(3)
        entries = [("layer0.q", torch.randn((24, 8), generator=g), 40, 105, 0, 2e-4),
                   ("layer0.down", torch.randn((16, 4), generator=g), 96, (1 << 40) + 7, 6, 1.5e-4)]
        payload = dp.pack_sync_payload(entries)
        np.save(os.path.join(out_dir, "sent.npy"), np.frombuffer(payload, dtype=np.uint8))
    got = dp.broadcast_sync_payload(payload, src=0)
    np.save(os.path.join(out_dir, f"got{rank}.npy"), np.frombuffer(got, dtype=np.uint8))
    torch.distributed.destroy_process_group()


def test_sync_payload_roundtrip_over_gloo(tmp_path):
    mp.spawn(_payload_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    sent = np.load(tmp_path / "sent.npy").tobytes()
    for r in range(2):
        assert np.load(tmp_path / f"got{r}.npy").tobytes() == sent
    dp = _load_dp()
    entries = dp.unpack_sync_payload(sent)
    assert [e[0] for e in entries] == ["layer0.q", "layer0.down"]
    name, S, k, seed, sid, ae = entries[1]
    assert S.shape == (16, 4) and k == 96 and seed == (1 << 40) + 7 and sid == 6 and ae == 1.5e-4
    g = torch.Generator().manual_seed(3)
    torch.randn((24, 8), generator=g)
    assert torch.equal(S, torch.randn((16, 4), generator=g))
    # O(d·r) + metadata, independent of k: the page's point
    assert len(sent) == dp.sync_payload_bytes([("layer0.q", 24, 8), ("layer0.down", 16, 4)])
    assert len(sent) < 4 * (24 * 8 + 16 * 4) + 200
    with pytest.raises(ValueError):
        dp.unpack_sync_payload(b"XXXX" + sent[4:])


def test_apply_sync_payload_batches_on_host(monkeypatch):
    # the apply groups the payload's entries by (r, αη) in order of first
    # appearance and hands each batch to one grouped merge; the merge calls
    # are recorded by a stand-in for the binding (no GPU library involved)
    import sys
    import types

    calls = []
    pkg = types.ModuleType("_fake_logra")
    pkg.__path__ = []
    binding = types.ModuleType("_fake_logra._binding")

    def plan(targets, r, stream=None):
        calls.append(("plan", r, [(tuple(t[0].shape), tuple(t[1].shape), t[2], t[3]) for t in targets]))
        return ("plan", r)

    binding.logra_merge_group_plan = plan
    binding.logra_merge_update_group = lambda p, ae, stream=None: calls.append(("launch", p[1], ae))
    binding.logra_merge_update = lambda W, S, seed, sid, r, ae, stream=None: calls.append(("single", r, ae, seed))
    monkeypatch.setitem(sys.modules, "_fake_logra", pkg)
    monkeypatch.setitem(sys.modules, "_fake_logra._binding", binding)
    spec = importlib.util.spec_from_file_location("_fake_logra.dp",
                                                  os.path.join(ROOT, "rank_gradient_sketching_gb300", "dp.py"))
    dp = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(dp)

    k = 32
    spec_e = [("a", 16, 4, 1e-2), ("b", 8, 16, 1e-2), ("c", 24, 4, 1e-2), ("d", 8, 4, 3e-2)]
    entries = [(n, torch.full((d, r), 0.5), k, 100 + j, j, ae) for j, (n, d, r, ae) in enumerate(spec_e)]
    weights = {n: torch.zeros((d, k), dtype=torch.bfloat16) for n, d, _, _ in spec_e}
    payload = dp.pack_sync_payload(entries)

    dp.apply_sync_payload(payload, weights)
    assert calls == [
        ("plan", 4, [((16, k), (16, 4), 100, 0), ((24, k), (24, 4), 102, 2)]), ("launch", 4, 1e-2),
        ("plan", 16, [((8, k), (8, 16), 101, 1)]), ("launch", 16, 1e-2),
        ("plan", 4, [((8, k), (8, 4), 103, 3)]), ("launch", 4, 3e-2),
    ]
    calls.clear()
    dp.apply_sync_payload(payload, weights, grouped=False)
    assert calls == [("single", 4, 1e-2, 100), ("single", 16, 1e-2, 101), ("single", 4, 1e-2, 102),
                     ("single", 4, 3e-2, 103)]
    with pytest.raises(ValueError):
        dp.apply_sync_payload(payload, {**weights, "b": torch.zeros((9, k), dtype=torch.bfloat16)})

    # A weight named twice (or two names for one tensor, as with tied
    # weights) must not sit in one launch: its CTAs would read and write the
    # same tiles.  The second entry opens a batch that runs after the first;
    # an independent entry joins the newest batch of its key.
    calls.clear()
    tied = torch.zeros((16, k), dtype=torch.bfloat16)
    spec_t = [("a", 16, 4, 1e-2), ("a_tied", 16, 4, 1e-2), ("c", 24, 4, 1e-2), ("a_rows", 8, 4, 1e-2)]
    w_t = {"a": tied, "a_tied": tied, "c": torch.zeros((24, k), dtype=torch.bfloat16),
           "a_rows": tied[4:12]}  # rows 4..11 of the tied weight: a partial overlap
    entries_t = [(n, torch.full((d, r), 0.5), k, 200 + j, j, ae) for j, (n, d, r, ae) in enumerate(spec_t)]
    dp.apply_sync_payload(dp.pack_sync_payload(entries_t), w_t)
    assert calls == [
        ("plan", 4, [((16, k), (16, 4), 200, 0)]), ("launch", 4, 1e-2),
        ("plan", 4, [((16, k), (16, 4), 201, 1), ((24, k), (24, 4), 202, 2)]), ("launch", 4, 1e-2),
        ("plan", 4, [((8, k), (8, 4), 203, 3)]), ("launch", 4, 1e-2),
    ]
