"""Data-parallel replicas (host-side gradient sum): the host reduction on CPU
with world_size-2 gloo process groups, and the replica step on the GPU with
two processes that meet only on the host."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    from host_memory_streamed_gb300 import replicas
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    g = torch.Generator().manual_seed(100 + rank)
    vals = (torch.randn(4099, generator=g) * 10.0 ** torch.randint(-6, 3, (4099,), generator=g)).to(torch.bfloat16)
    raw = vals.view(torch.uint8).clone()
    replicas.allreduce_mean_bf16_(raw)
    torch.save(raw.view(torch.bfloat16).clone(), os.path.join(out_dir, f"r{rank}.pt"))
    dist.destroy_process_group()


def test_allreduce_mean_bf16_two_ranks(tmp_path):
    """Both ranks end with the same BF16 values: (a + b) / 2 summed in FP32
    and rounded once."""
    world, port = 2, _free_port()
    mp.start_processes(_reduce_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    r0, r1 = torch.load(tmp_path / "r0.pt"), torch.load(tmp_path / "r1.pt")
    assert torch.equal(r0.view(torch.int16), r1.view(torch.int16))
    vals = []
    for rank in range(world):
        g = torch.Generator().manual_seed(100 + rank)
        vals.append((torch.randn(4099, generator=g) * 10.0 ** torch.randint(-6, 3, (4099,), generator=g))
                    .to(torch.bfloat16).to(torch.float32))
    expect = ((vals[0] + vals[1]) / 2).to(torch.bfloat16)
    assert torch.equal(r0.view(torch.int16), expect.view(torch.int16))


def _replica_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    import host_memory_streamed_gb300 as hms
    import mt_inputs
    from host_memory_streamed_gb300 import replicas
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    s = mt_inputs.PRESETS["tiny"]
    m = hms.StreamedDecoder.from_shape(s, device="cuda:0")
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    loss = replicas.replica_step(m, mt_inputs.step_tokens(s, 1 + rank))
    torch.save({"loss": loss, "w": m.weights(), "g": m.grads(), "mv": m.moments(), "step": m.step},
               os.path.join(out_dir, f"rep{rank}.pt"))
    m.close()
    dist.destroy_process_group()


@pytest.mark.gpu
def test_two_replicas_match_oracle_on_the_global_batch(tmp_path):
    """Two replicas (two processes on one GPU, synchronised only through the
    host all-reduce) on the step-1 and step-2 token batches: the same weights
    on both, the averaged gradient is the oracle's for the concatenated batch,
    and Adam on it matches the oracle's update."""
    import mt_inputs
    import oracle
    from oracle import OracleConfig
    from tests import parity
    world, port = 2, _free_port()
    mp.start_processes(_replica_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    r = [torch.load(tmp_path / f"rep{k}.pt") for k in range(world)]
    for (n, a), (_, b) in zip(parity.flat_named(r[0]["w"]), parity.flat_named(r[1]["w"])):
        assert torch.equal(a, b), n
    assert r[0]["loss"] == r[1]["loss"] and r[0]["step"] == r[1]["step"] == 1
    s = mt_inputs.PRESETS["tiny"]
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = torch.cat([mt_inputs.step_tokens(s, 1), mt_inputs.step_tokens(s, 2)])
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    assert abs(r[0]["loss"] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r[0]["g"], grads)
    m, v = r[0]["mv"]
    parity.assert_adam_matches(r[0]["w"], params, r[0]["g"], m, v, 1, cfg)
