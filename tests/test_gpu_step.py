"""GPU training step through the C-ABI against the CPU oracle, and the
schedule's bit-exact self-consistency (streamed == resident, recompute ==
stored activations, K=1 == K=2 == no double buffer, repeat runs, resume)."""
import pytest
import torch

import mt_inputs
import oracle
from oracle import OracleConfig
from tests import parity

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")


def _run(shape, steps=1, flags=0, jitter=0.1, **kw):
    m = hms.StreamedDecoder.from_shape(shape, flags=flags, **kw)
    params = mt_inputs.model_weights(shape, gain_jitter=jitter)
    m.load_weights(params)
    out = {"params0": params, "loss": [], "w": [], "g": [], "mv": []}
    for n in range(1, steps + 1):
        out["loss"].append(m.train_step(mt_inputs.step_tokens(shape, n)))
        out["w"].append(m.weights())
        out["g"].append(m.grads())
        out["mv"].append(m.moments())
    out["stats"] = m.stats()
    m.close()
    return out


def _equal_trees(a, b):
    for (n, x), (_, y) in zip(parity.flat_named(a), parity.flat_named(b)):
        assert torch.equal(x, y), n


SHAPES = {
    "tiny": mt_inputs.PRESETS["tiny"],
    # GQA, head_dim 128, ragged sequence (not a multiple of 64/128), 3 layers
    "gqa128": mt_inputs.PRESETS["tiny"].with_(n_layers=3, d_model=256, n_heads=4, n_kv_heads=2, head_dim=128,
                                              ffn=344, vocab=520, batch=2, seq=180),
}


@pytest.mark.parametrize("name", ["tiny", "gqa128"])
def test_step_matches_oracle(name):
    s = SHAPES[name]
    cfg = OracleConfig.from_shape(s)
    r = _run(s)
    tokens = mt_inputs.step_tokens(s, 1)
    loss, grads = oracle.model_loss_and_grads(r["params0"], tokens, cfg)
    assert abs(r["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r["g"][0], grads)
    m, v = r["mv"][0]
    parity.assert_adam_matches(r["w"][0], r["params0"], r["g"][0], m, v, 1, cfg)
    ok, total, excluded, worst = parity.adam_vs_oracle_grads(r["w"][0], r["params0"], grads, 1, cfg)
    assert ok >= 0.99 * total, (ok, total, worst[:5])


def test_three_step_loss_trajectory_matches_oracle():
    s = SHAPES["tiny"]
    cfg = OracleConfig.from_shape(s)
    r = _run(s, steps=3)
    params, state = r["params0"], None
    for n in range(1, 4):
        tok = mt_inputs.step_tokens(s, n)
        loss, grads, params, state = oracle.train_step(params, state, tok, n, cfg)
        assert abs(r["loss"][n - 1] - loss) <= parity.LOSS_RTOL * abs(loss), (n, r["loss"][n - 1], loss)
        parity.assert_grads_close(r["g"][n - 1], grads)
        # embedding rows of token ids absent from this step hold exactly zero
        untouched = torch.ones(s.vocab, dtype=torch.bool)
        untouched[tok[:, :-1].reshape(-1).long()] = False
        assert torch.all(r["g"][n - 1]["embed"]["E"][untouched] == 0)


def test_streamed_equals_resident_bitexact():
    s = SHAPES["gqa128"]
    a = _run(s, steps=2)
    b = _run(s, steps=2, flags=hms.MT_RESIDENT)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    _equal_trees(a["g"][-1], b["g"][-1])


def test_recompute_equals_stored_activations_bitexact():
    s = SHAPES["gqa128"]
    a = _run(s, steps=2)
    b = _run(s, steps=2, flags=hms.MT_STORE_ACTS)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    _equal_trees(a["g"][-1], b["g"][-1])


@pytest.mark.parametrize("K,keep", [(1, 1), (1, 2), (2, 1), (2, 2), (3, 2), (1, 3)])
def test_kept_layers_equal_recompute_bitexact(K, keep):
    """The last `keep` layers keep their internals from the forward (no
    recompute in their backward); the result is the recompute schedule's, bit
    for bit, and the executed-FLOP count drops by their internal recompute."""
    s = SHAPES["gqa128"].with_(ckpt_every=K)
    a = _run(s, steps=2)
    b = _run(s, steps=2, keep_layers=keep)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    _equal_trees(a["g"][-1], b["g"][-1])
    assert b["stats"]["flops_executed"] < a["stats"]["flops_executed"]


@pytest.mark.parametrize("name,keep", [("tiny", 0), ("gqa128", 3)])
def test_async_adam_equals_synchronous_bitexact(name, keep):
    """MT_ASYNC_ADAM lets a step return while its Adam updates still run; the
    next step waits per tile, reads wait too, so three steps give the
    synchronous step's weights, gradients and moments bit for bit."""
    s = SHAPES[name]
    a = _run(s, steps=3, keep_layers=keep)
    b = _run(s, steps=3, flags=hms.MT_ASYNC_ADAM, keep_layers=keep)
    assert a["loss"] == b["loss"]
    for n in range(3):
        _equal_trees(a["w"][n], b["w"][n])
        _equal_trees(a["g"][n], b["g"][n])
        for x, y in zip(a["mv"][n], b["mv"][n]):
            _equal_trees(x, y)


@pytest.mark.parametrize("name,flags,keep", [("tiny", 0, 0), ("gqa128", hms.MT_ASYNC_ADAM, 3),
                                             ("tiny", hms.MT_TIE_EMBEDDINGS, 0)])
def test_direct_gradient_landing_equals_slab_path_bitexact(name, flags, keep):
    """MT_DIRECT_GRADS: gradient chunks land straight in the page-locked G
    sections (no slab copy); weights, gradients and moments are the slab
    path's bit for bit over three steps."""
    s = SHAPES[name]
    a = _run(s, steps=3, flags=flags, keep_layers=keep)
    b = _run(s, steps=3, flags=flags | hms.MT_DIRECT_GRADS, keep_layers=keep)
    assert a["loss"] == b["loss"]
    for n in range(3):
        _equal_trees(a["w"][n], b["w"][n])
        _equal_trees(a["g"][n], b["g"][n])
        for x, y in zip(a["mv"][n], b["mv"][n]):
            _equal_trees(x, y)


@pytest.mark.parametrize("name,flags,keep", [("tiny", 0, 0),
                                             ("gqa128", hms.MT_ASYNC_ADAM | hms.MT_DIRECT_GRADS, 3),
                                             ("tiny", hms.MT_TIE_EMBEDDINGS | hms.MT_DIRECT_GRADS, 0)])
def test_direct_weight_upload_equals_staged_path_bitexact(name, flags, keep):
    """MT_DIRECT_WEIGHTS: each upload's DMA reads the page-locked W section in
    place, in chunks smaller than a tile; losses, weights, gradients and
    moments are the staged path's bit for bit over three steps (so every
    upload read the weights after that tile's previous Adam update)."""
    s = SHAPES[name]
    a = _run(s, steps=3, flags=flags, keep_layers=keep, stage_bytes=48 << 10)
    b = _run(s, steps=3, flags=flags | hms.MT_DIRECT_WEIGHTS, keep_layers=keep, stage_bytes=48 << 10)
    assert a["loss"] == b["loss"]
    for n in range(3):
        _equal_trees(a["w"][n], b["w"][n])
        _equal_trees(a["g"][n], b["g"][n])
        for x, y in zip(a["mv"][n], b["mv"][n]):
            _equal_trees(x, y)


def test_direct_gradient_landing_nonfinite_step_updates_nothing():
    """A non-finite value in the forward (an infinite weight) with direct
    gradient landing: MT_ENONFINITE and no weight updated."""
    s = SHAPES["tiny"]
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    params["layers"][0]["wq"][0, 0] = float("inf")
    m = hms.StreamedDecoder.from_shape(s, flags=hms.MT_DIRECT_GRADS)
    m.load_weights(params)
    with pytest.raises(hms.MtError) as e:
        m.train_step(mt_inputs.step_tokens(s, 1))
    assert e.value.code == hms._lib.MT_ENONFINITE
    _equal_trees(m.weights(), params)
    m.close()


def test_direct_gradient_landing_with_micro_batches_matches_oracle():
    """The first micro-batch lands directly, the second adds through the slabs."""
    s = SHAPES["gqa128"]
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    t1, t2 = mt_inputs.step_tokens(s, 1), mt_inputs.step_tokens(s, 2)
    m = hms.StreamedDecoder.from_shape(s, flags=hms.MT_DIRECT_GRADS | hms.MT_ASYNC_ADAM)
    m.load_weights(params)
    loss = m.train_step_micro(torch.stack([t1, t2]))
    g, w = m.grads(), m.weights()
    mm, vv = m.moments()
    m.close()
    loss_ref, grads = oracle.model_loss_and_grads(params, torch.cat([t1, t2]), cfg)
    assert abs(loss - loss_ref) <= parity.LOSS_RTOL * abs(loss_ref)
    parity.assert_grads_close(g, grads)
    parity.assert_adam_matches(w, params, g, mm, vv, 1, cfg)


@pytest.mark.parametrize("direct_weights", [0, hms.MT_DIRECT_WEIGHTS])
def test_timeline_spans_every_visit_and_chunk_copy(direct_weights):
    """mt_get_timeline: one compute span per visit and one span per chunk copy
    in each direction, each with t1 >= t0; the copies of a visit's weights
    end before that visit's compute starts (Weights-Ready)."""
    s = SHAPES["gqa128"]
    stage, slab = 64 << 10, 32 << 10
    flags = hms.MT_TIME_KERNELS | hms.MT_DIRECT_GRADS | direct_weights
    m = hms.StreamedDecoder.from_shape(s, flags=flags, stage_bytes=stage,
                                       grad_slab_bytes=slab, n_grad_slabs=4)
    m.load_weights(mt_inputs.model_weights(s))
    m.train_step(mt_inputs.step_tokens(s, 1))
    tl = m.timeline()
    plan = hms.plan_schedule(s.n_layers, s.ckpt_every)
    m.close()
    L = hms._lib
    comp = [x for x in tl if x[0] == L.SPAN_COMPUTE]
    h2d = [x for x in tl if x[0] == L.SPAN_H2D]
    d2h = [x for x in tl if x[0] == L.SPAN_D2H]
    assert len(comp) == len(plan)
    wb = [info["w_bytes"] for info in m.infos]
    assert len(h2d) == sum(-(-wb[v["tile"]] // stage) for v in plan if v["h2d"])
    layer_grads = [v for v in plan if v["kind"] in (L.VISIT_LAYER_BWD, L.VISIT_HEAD)]
    assert len(d2h) >= sum(-(-wb[v["tile"]] // slab) for v in layer_grads)
    assert all(t1 >= t0 for _, _, t0, t1 in tl)
    start = {v: t0 for k, v, t0, _ in comp}
    for _, v, _, t1 in h2d:
        assert t1 <= start[v] + 1e-3, v


@pytest.mark.parametrize("variant", ["ckpt2", "ckpt3", "single_buffer", "small_chunks"])
def test_schedule_variants_bitexact(variant):
    s = SHAPES["gqa128"]
    a = _run(s, steps=2)
    if variant == "ckpt2":
        b = _run(s.with_(ckpt_every=2), steps=2)
    elif variant == "ckpt3":
        b = _run(s.with_(ckpt_every=3), steps=2)
    elif variant == "single_buffer":
        b = _run(s, steps=2, flags=hms.MT_NO_DOUBLE_BUFFER)
    else:  # many staging chunks and gradient slabs per tile, 2 slabs only
        b = _run(s, steps=2, stage_bytes=64 << 10, grad_slab_bytes=32 << 10, n_grad_slabs=2, n_pack_threads=3)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    _equal_trees(a["g"][-1], b["g"][-1])


def test_repeat_runs_bitexact():
    s = SHAPES["tiny"]
    a = _run(s, steps=2)
    b = _run(s, steps=2)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    for x, y in zip(a["mv"][-1], b["mv"][-1]):
        _equal_trees(x, y)


def test_save_reload_continue_bitexact():
    s = SHAPES["tiny"]
    full = _run(s, steps=3)
    m = hms.StreamedDecoder.from_shape(s)
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    m.train_step(mt_inputs.step_tokens(s, 1))
    saved = [[m.get_tile(i, p) for p in range(4)] for i in range(m.n_tiles)]
    step = m.step
    m.close()
    m2 = hms.StreamedDecoder.from_shape(s)
    for i in range(m2.n_tiles):
        for p in range(4):
            m2.load_tile(i, p, saved[i][p])
    m2.step = step
    l2 = m2.train_step(mt_inputs.step_tokens(s, 2))
    l3 = m2.train_step(mt_inputs.step_tokens(s, 3))
    assert [l2, l3] == full["loss"][1:]
    _equal_trees(m2.weights(), full["w"][-1])
    m2.close()


def test_statistics_account_for_streamed_bytes():
    s = SHAPES["gqa128"]
    r = _run(s, steps=1)
    st = r["stats"]
    m = hms.StreamedDecoder.from_shape(s)
    infos = m.infos
    m.close()
    layer_w = infos[1]["w_bytes"]
    # K = 1: every layer is streamed for forward and again for backward, except
    # the last layer, whose weights are still resident when backward starts.
    expect_h2d = infos[0]["w_bytes"] + infos[-1]["w_bytes"] + (2 * s.n_layers - 1) * layer_w
    assert st["h2d_bytes"] == expect_h2d
    # gradients: every layer tile and the head whole; the embedding only for the
    # token ids that occur in the step (its other rows are zero)
    distinct = int(torch.unique(mt_inputs.step_tokens(s, 1)[:, :-1]).numel())
    assert st["d2h_bytes"] == sum(i["w_bytes"] for i in infos[1:]) + 2 * distinct * s.d_model
    assert st["step"] == 1 and st["gemm_launches"] > 0


@pytest.mark.parametrize("K", [1, 2])
def test_executed_flops_are_the_launched_gemms_plus_attention(K):
    """flops_executed counts what the schedule launches: every GEMM launch
    (2*M*N*K each, recorded per launch under MT_TIME_KERNELS) plus causal
    attention once per forward visit, boundary recompute and backward visit's
    internal recompute, and twice per layer backward."""
    s = SHAPES["gqa128"].with_(ckpt_every=K)
    st = _run(s, flags=hms.MT_TIME_KERNELS)["stats"]
    plan = hms.plan_schedule(s.n_layers, K)
    kinds = (hms._lib.VISIT_LAYER_FWD, hms._lib.VISIT_RECOMPUTE, hms._lib.VISIT_LAYER_BWD)
    n_attn = sum(1 for v in plan if v["kind"] in kinds) + 2 * s.n_layers
    attn = 4.0 * s.batch * s.n_heads * s.head_dim * s.seq * (s.seq + 1) / 2
    assert st["gemm_launches"] > 0
    assert st["flops_executed"] == pytest.approx(st["gemm_flops"] + n_attn * attn, rel=1e-9)


def test_nonfinite_loss_skips_every_update():
    """A non-finite loss is seen before any gradient lands: the step reports
    MT_ENONFINITE and no weight is updated."""
    s = SHAPES["tiny"]
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    params["head"]["wh"][3, 5] = float("inf")
    m = hms.StreamedDecoder.from_shape(s)
    m.load_weights(params)
    with pytest.raises(hms.MtError) as e:
        m.train_step(mt_inputs.step_tokens(s, 1))
    assert e.value.code == hms._lib.MT_ENONFINITE
    _equal_trees(m.weights(), params)
    m.close()


def test_chunked_mlp_matches_oracle_and_repeats():
    """The MLP over row chunks (long-sequence mode: 128-row chunks of a
    360-token step, the last one ragged) against the oracle, and bit-exact
    across repeat runs."""
    s = SHAPES["gqa128"]
    cfg = OracleConfig.from_shape(s)
    r = _run(s, mlp_chunk_rows=128)
    tokens = mt_inputs.step_tokens(s, 1)
    loss, grads = oracle.model_loss_and_grads(r["params0"], tokens, cfg)
    assert abs(r["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r["g"][0], grads)
    m, v = r["mv"][0]
    parity.assert_adam_matches(r["w"][0], r["params0"], r["g"][0], m, v, 1, cfg)
    r2 = _run(s, mlp_chunk_rows=128)
    assert r["loss"] == r2["loss"]
    _equal_trees(r["g"][0], r2["g"][0])
    _equal_trees(r["w"][0], r2["w"][0])


def test_micro_batch_accumulation_matches_oracle():
    """Two micro-batches in one step: the loss and every gradient are those of
    the mean over both micro-batches' targets (the oracle on the concatenated
    batch), and Adam runs once on the accumulated gradient."""
    s = SHAPES["gqa128"]
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    t1, t2 = mt_inputs.step_tokens(s, 1), mt_inputs.step_tokens(s, 2)
    m = hms.StreamedDecoder.from_shape(s)
    m.load_weights(params)
    loss = m.train_step_micro(torch.stack([t1, t2]))
    g, w = m.grads(), m.weights()
    mm, vv = m.moments()
    assert m.step == 1
    m.close()
    loss_ref, grads = oracle.model_loss_and_grads(params, torch.cat([t1, t2]), cfg)
    assert abs(loss - loss_ref) <= parity.LOSS_RTOL * abs(loss_ref)
    parity.assert_grads_close(g, grads)
    parity.assert_adam_matches(w, params, g, mm, vv, 1, cfg)


def test_one_micro_batch_is_the_plain_step():
    s = SHAPES["tiny"]
    a = _run(s, steps=1)
    m = hms.StreamedDecoder.from_shape(s)
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    loss = m.train_step_micro(mt_inputs.step_tokens(s, 1)[None])
    assert loss == a["loss"][0]
    _equal_trees(m.weights(), a["w"][0])
    _equal_trees(m.grads(), a["g"][0])
    m.close()


# ------------------------------------------------------------------ tied embeddings
def _run_tied(shape, tokens_list, flags=0, micro=False):
    m = hms.StreamedDecoder.from_shape(shape, flags=flags | hms.MT_TIE_EMBEDDINGS)
    assert m.n_tiles == shape.n_layers + 1
    params = mt_inputs.tied(mt_inputs.model_weights(shape, gain_jitter=0.1))
    m.load_weights(params)
    out = {"params0": params, "loss": [], "w": [], "g": [], "mv": []}
    for tok in tokens_list:
        out["loss"].append(m.train_step_micro(tok) if micro else m.train_step(tok))
        out["w"].append(m.weights())
        out["g"].append(m.grads())
        out["mv"].append(m.moments())
    m.close()
    return out


@pytest.mark.parametrize("name", ["tiny", "one_layer", "gqa128"])
def test_tied_embeddings_step_matches_oracle(name):
    """MT_TIE_EMBEDDINGS: one host tile for E and the final gain; the head
    streams it and uses E as W_h, E's gradient is the head's plus the
    embedding's, Adam updates every row once.  With one layer the head's
    visit finds the embedding tile still in a device buffer (no second
    upload); with more layers it is streamed again."""
    s = SHAPES["tiny"].with_(n_layers=1) if name == "one_layer" else SHAPES[name]
    cfg = OracleConfig.from_shape(s)
    tokens = mt_inputs.step_tokens(s, 1)
    r = _run_tied(s, [tokens])
    assert set(r["g"][0]["head"]) == {"gf"} and set(r["w"][0]["head"]) == {"gf"}
    loss, grads = oracle.model_loss_and_grads(r["params0"], tokens, cfg)
    assert abs(r["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r["g"][0], grads)
    m, v = r["mv"][0]
    parity.assert_adam_matches(r["w"][0], r["params0"], r["g"][0], m, v, 1, cfg)
    # rows of token ids absent from the step carry the head's gradient alone
    untouched = torch.ones(s.vocab, dtype=torch.bool)
    untouched[tokens[:, :-1].reshape(-1).long()] = False
    assert int(untouched.sum()) > 0
    assert torch.any(r["g"][0]["embed"]["E"][untouched] != 0)


def test_tied_embeddings_trajectory_and_resident_bitexact():
    s = SHAPES["gqa128"]
    cfg = OracleConfig.from_shape(s)
    toks = [mt_inputs.step_tokens(s, n) for n in (1, 2)]
    a = _run_tied(s, toks)
    b = _run_tied(s, toks, flags=hms.MT_RESIDENT)
    assert a["loss"] == b["loss"]
    _equal_trees(a["w"][-1], b["w"][-1])
    _equal_trees(a["g"][-1], b["g"][-1])
    params, state = a["params0"], None
    for n, tok in enumerate(toks, 1):
        loss, grads, params, state = oracle.train_step(params, state, tok, n, cfg)
        assert abs(a["loss"][n - 1] - loss) <= parity.LOSS_RTOL * abs(loss), (n, a["loss"][n - 1], loss)
        parity.assert_grads_close(a["g"][n - 1], grads)


def test_tied_embeddings_micro_batches_match_oracle():
    s = SHAPES["gqa128"]
    cfg = OracleConfig.from_shape(s)
    t1, t2 = mt_inputs.step_tokens(s, 1), mt_inputs.step_tokens(s, 2)
    r = _run_tied(s, [torch.stack([t1, t2])], micro=True)
    loss_ref, grads = oracle.model_loss_and_grads(r["params0"], torch.cat([t1, t2]), cfg)
    assert abs(r["loss"][0] - loss_ref) <= parity.LOSS_RTOL * abs(loss_ref)
    parity.assert_grads_close(r["g"][0], grads)
    m, v = r["mv"][0]
    parity.assert_adam_matches(r["w"][0], r["params0"], r["g"][0], m, v, 1, cfg)



def test_grads_only_then_adam_is_the_plain_step():
    """mt_train_step_grads + mt_apply_adam (the data-parallel replica split)
    reproduce mt_train_step bit for bit: loss, weights, gradients, moments."""
    s = SHAPES["gqa128"]
    a = _run(s, steps=2)
    m = hms.StreamedDecoder.from_shape(s)
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    for n in (1, 2):
        assert m.train_step_grads(mt_inputs.step_tokens(s, n)) == a["loss"][n - 1]
        assert m.step == n - 1
        m.apply_adam()
    assert m.step == 2
    _equal_trees(m.weights(), a["w"][-1])
    _equal_trees(m.grads(), a["g"][-1])
    for x, y in zip(m.moments(), a["mv"][-1]):
        _equal_trees(x, y)
    m.close()


def test_visit_log_prints_one_line_per_visit(capfd):
    """MT_VISIT_LOG: after the step, one '[mt visit]' line per visit of the
    schedule (embedding, L layers forward, head, L layers backward, embedding
    backward at K = 1) and the host-tail line, on stderr."""
    s = SHAPES["tiny"]
    m = hms.StreamedDecoder.from_shape(s, flags=hms.MT_VISIT_LOG)
    m.load_weights(mt_inputs.model_weights(s, gain_jitter=0.1))
    capfd.readouterr()
    m.train_step(mt_inputs.step_tokens(s, 1))
    m.close()
    err = capfd.readouterr().err.splitlines()
    visits = [l for l in err if l.startswith("[mt visit]") and " gap " in l]
    tails = [l for l in err if l.startswith("[mt visit] compute stream ends")]
    assert len(visits) == 2 * s.n_layers + 3, err[:5]
    assert len(tails) == 1
    assert "layer_bwd" in visits[-2] and "embed_bwd" in visits[-1]
