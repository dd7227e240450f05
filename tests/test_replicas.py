"""Data-parallel replicas of one model (a replica group): config checks and
the agreement on a group name with world_size-2 gloo process groups on the
CPU; on the GPU, groups of two processes (both on the one device, meeting
only in host shared memory, no kernel waiting on another process) checked
bit for bit against one model's micro-batch step, against the oracle, and for
failure and non-finite propagation."""
import ctypes as C
import os
import socket
import time

import pytest
import torch
import torch.multiprocessing as mp

import mt_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SHAPES = {
    "tiny": mt_inputs.PRESETS["tiny"],
    # GQA, head_dim 128, ragged sequence, 3 layers
    "gqa128": mt_inputs.PRESETS["tiny"].with_(n_layers=3, d_model=256, n_heads=4, n_kv_heads=2, head_dim=128,
                                              ffn=344, vocab=520, batch=2, seq=180),
    # mixture-of-experts layers: 8 experts, top-2, grouped expert GEMMs
    "moe": mt_inputs.PRESETS["tiny"].with_(n_experts=8, top_k=2, ffn=136),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tokens(s, step, rank):
    return mt_inputs.step_tokens(s, 10 * step + rank + 1)


# ------------------------------------------------------------------ CPU
def _cfg(shape, **kw):
    from host_memory_streamed_gb300 import _lib
    c = _lib.MtConfig()
    for k in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "batch", "seq",
              "ckpt_every", "rms_eps", "rope_theta", "lr", "beta1", "beta2", "adam_eps", "weight_decay"):
        setattr(c, k, getattr(shape, k))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("bad,msg", [
    (dict(n_replicas=65, replica_rank=0, replica_name=b"g"), "n_replicas"),
    (dict(n_replicas=-1), "n_replicas"),
    (dict(n_replicas=2, replica_rank=2, replica_name=b"g"), "replica_rank"),
    (dict(n_replicas=2, replica_rank=-1, replica_name=b"g"), "replica_rank"),
    (dict(n_replicas=2, replica_rank=0, replica_name=b""), "replica_name"),
    (dict(n_replicas=2, replica_rank=0, replica_name=b"a/b"), "replica_name"),
    (dict(n_replicas=2, replica_rank=1, replica_name=b"g", flags=1), "MT_RESIDENT"),
    (dict(n_replicas=2, replica_rank=1, replica_name=b"g", flags=128), "MT_TIE_EMBEDDINGS"),
])
def test_group_config_rejections(bad, msg):
    from host_memory_streamed_gb300 import _lib, build
    build.build()
    lib = _lib.lib()
    assert lib.mt_required_device_bytes(C.byref(_cfg(SHAPES["tiny"], **bad))) == -1
    assert msg in lib.mt_last_error(None).decode()


def test_group_config_accepted_and_sized_as_a_single_model():
    """A replica's device arena is that of a model of its own: the group only
    moves the host tiles into shared memory."""
    from host_memory_streamed_gb300 import _lib, build
    build.build()
    lib = _lib.lib()
    s = SHAPES["gqa128"]
    one = lib.mt_required_device_bytes(C.byref(_cfg(s)))
    rep = lib.mt_required_device_bytes(C.byref(_cfg(s, n_replicas=8, replica_rank=7, replica_name=b"mt.g-1_x")))
    assert one > 0 and rep == one


def _name_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    from host_memory_streamed_gb300 import replicas
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    names = [replicas.shared_group_name(), replicas.shared_group_name()]
    torch.save(names, os.path.join(out_dir, f"n{rank}.pt"))
    dist.destroy_process_group()


def test_group_name_agreed_over_a_gloo_group(tmp_path):
    """Every rank of a process group gets replica 0's name; two calls give two
    names; each is a valid shared-memory name."""
    world, port = 2, _free_port()
    mp.start_processes(_name_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    n0, n1 = torch.load(tmp_path / "n0.pt"), torch.load(tmp_path / "n1.pt")
    assert n0 == n1 and n0[0] != n0[1]
    for n in n0:
        assert 0 < len(n) < 48 and all(ch.isalnum() or ch in "_-." for ch in n)


# ------------------------------------------------------------------ GPU
def _group_worker(rank, n, name, out_dir, case):
    import host_memory_streamed_gb300 as hms
    from host_memory_streamed_gb300 import replicas
    s = SHAPES[case["shape"]]
    out = {"loss": [], "w": [], "g": [], "mv": [], "err": None, "err_s": None}
    m = None
    try:
        m = replicas.open_replica(s, name, rank, n, device="cuda:0", flags=case.get("flags", 0),
                                  keep_layers=case.get("keep", 0), timeout_ms=case.get("timeout_ms", 0),
                                  grad_slab_bytes=case.get("slab", 0), stage_bytes=case.get("stage", 0))
        if rank == 0:
            params = mt_inputs.model_weights(s, gain_jitter=0.1)
            if case.get("inf"):
                params["layers"][0]["wq"][0, 0] = float("inf")
            m.load_weights(params)
        m.barrier()
        if case.get("inject") is not None and rank == case["inject_rank"]:
            m.debug_inject(case["inject"], 0)
        for k in range(case["steps"]):
            t0 = time.monotonic()
            try:
                out["loss"].append(replicas.replica_step(m, _tokens(s, k, rank)))
            except hms.MtError as e:
                out["err"], out["err_s"], out["msg"] = e.code, time.monotonic() - t0, str(e)
                if e.code == hms._lib.MT_ENONFINITE and rank == 0:
                    m.sync()
                    out["w_after"] = m.weights()
                break
            if rank == 0 or case.get("all_read"):
                m.sync()
                out["w"].append(m.weights())
                out["g"].append(m.grads())
                out["mv"].append(m.moments())
            m.barrier()  # no replica starts the next step while another reads the tiles
        if out["err"] is None:
            m.sync()
            out["step"] = m.step
            m.barrier()  # no replica leaves while another still reads the tiles
    finally:
        torch.save(out, os.path.join(out_dir, f"g{rank}.pt"))
        if m is not None:
            m.close()


def _run_group(tmp_path, case, n=2):
    from host_memory_streamed_gb300 import replicas
    name = replicas.group_name("mt-test")
    mp.start_processes(_group_worker, args=(n, name, str(tmp_path), case), nprocs=n, start_method="spawn")
    return [torch.load(tmp_path / f"g{r}.pt") for r in range(n)]


def _equal_trees(a, b):
    from tests import parity
    for (n, x), (_, y) in zip(parity.flat_named(a), parity.flat_named(b)):
        assert torch.equal(x, y), n


CASES = {
    "tiny": dict(shape="tiny", steps=3),
    # several chunks per tile (small slabs and staging chunks), kept layers,
    # asynchronous Adam, direct gradient landing on replica 0, weights read in place
    "gqa128-async-direct": dict(shape="gqa128", steps=3, keep=3, slab=32 << 10, stage=48 << 10, all_read=True,
                                flags=256 | 512 | 1024),
    "moe-async-direct": dict(shape="moe", steps=2, flags=256 | 512 | 1024),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", list(CASES))
def test_group_equals_micro_batch_step_bitexact(tmp_path, case):
    """Two replicas, three group steps: every loss, and the weights, gradients
    and moments after every step, equal one model's train_step_micro over
    the two replicas' batches in rank order, bit for bit; both replicas read
    the same tiles."""
    import host_memory_streamed_gb300 as hms
    c = CASES[case]
    r = _run_group(tmp_path, c)
    assert r[0]["err"] is None and r[1]["err"] is None, (r[0].get("msg"), r[1].get("msg"))
    assert r[0]["loss"] == r[1]["loss"] and r[0]["step"] == r[1]["step"] == c["steps"]
    s = SHAPES[c["shape"]]
    m = hms.StreamedDecoder.from_shape(s, flags=c.get("flags", 0), keep_layers=c.get("keep", 0),
                                       grad_slab_bytes=c.get("slab", 0), stage_bytes=c.get("stage", 0))
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    for k in range(c["steps"]):
        loss = m.train_step_micro(torch.stack([_tokens(s, k, 0), _tokens(s, k, 1)]))
        assert loss == r[0]["loss"][k], k
        w, g, mv = m.weights(), m.grads(), m.moments()
        _equal_trees(w, r[0]["w"][k])
        _equal_trees(g, r[0]["g"][k])
        for x, y in zip(mv, r[0]["mv"][k]):
            _equal_trees(x, y)
        if c.get("all_read"):
            _equal_trees(w, r[1]["w"][k])
    m.close()


@pytest.mark.gpu
def test_group_matches_oracle_on_the_global_batch(tmp_path):
    """Two replicas, one step: the loss and the summed gradient are the
    oracle's for the concatenated batch, and Adam on it matches the oracle's
    update."""
    import oracle
    from oracle import OracleConfig
    from tests import parity
    r = _run_group(tmp_path, dict(shape="tiny", steps=1))
    assert r[0]["err"] is None and r[1]["err"] is None
    s = SHAPES["tiny"]
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = torch.cat([_tokens(s, 0, 0), _tokens(s, 0, 1)])
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    assert abs(r[0]["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r[0]["g"][0], grads)
    m, v = r[0]["mv"][0]
    parity.assert_adam_matches(r[0]["w"][0], params, r[0]["g"][0], m, v, 1, cfg)


@pytest.mark.gpu
def test_group_failure_reaches_the_other_replica(tmp_path):
    """Replica 1's loader fails (host-side injection) in the first step:
    replica 1 reports it, and replica 0 stops with MT_EINTERNAL naming the
    group long before its 30 s wait bound."""
    from host_memory_streamed_gb300 import _lib
    r = _run_group(tmp_path, dict(shape="tiny", steps=1, inject=_lib.MT_INJECT_LOADER_FAIL, inject_rank=1,
                                  timeout_ms=30000))
    assert r[1]["err"] == _lib.MT_EINTERNAL and "injected loader" in r[1]["msg"], r[1].get("msg")
    assert r[0]["err"] == _lib.MT_EINTERNAL and "another replica" in r[0]["msg"], r[0].get("msg")
    assert r[0]["err_s"] < 15.0


@pytest.mark.gpu
def test_group_nonfinite_step_updates_nothing(tmp_path):
    """An infinite weight: every replica returns MT_ENONFINITE and no weight
    changes."""
    from host_memory_streamed_gb300 import _lib
    r = _run_group(tmp_path, dict(shape="tiny", steps=1, inf=True))
    assert r[0]["err"] == r[1]["err"] == _lib.MT_ENONFINITE
    params = mt_inputs.model_weights(SHAPES["tiny"], gain_jitter=0.1)
    params["layers"][0]["wq"][0, 0] = float("inf")
    _equal_trees(r[0]["w_after"], params)
