"""The streamed visit order of one training step (``mt_plan_schedule``), on
the CPU, against the method's description: every layer forward in order, the
head, then the checkpoint blocks in reverse with block recompute (layers
s .. e-2 run forward again from the checkpoint x_s, then layers e-1 .. s
backward; MegaTrain paperlayer.ai summary, §3 "Execution workflow" and §A.3
"Block-wise recomputation"), then the embedding gradient; two device weight
buffers used in ping-pong (the next tile streams into the buffer the current
visit does not compute on, after its Buffer-Free event), and a tile still held
by a buffer not streamed again."""
import pytest

import host_memory_streamed_gb300 as hms
from host_memory_streamed_gb300 import _lib

EF, LF, HD, RC, LB, EB = (_lib.VISIT_EMBED_FWD, _lib.VISIT_LAYER_FWD, _lib.VISIT_HEAD, _lib.VISIT_RECOMPUTE,
                          _lib.VISIT_LAYER_BWD, _lib.VISIT_EMBED_BWD)


@pytest.fixture(scope="module", autouse=True)
def built():
    from host_memory_streamed_gb300 import build
    build.build()


def expected_order(L, K, store_acts=False, keep=0):
    """(kind, layer) of every visit, written out from the description: the
    kept layers (the last `keep`, or all with stored activations) go backward
    without recompute, the others in checkpoint blocks of K."""
    v = [(EF, -1)] + [(LF, i) for i in range(L)] + [(HD, -1)]
    L0 = 0 if store_acts else max(0, L - keep)
    v += [(LB, j) for j in range(L - 1, L0 - 1, -1)]
    starts = list(range(0, L0, K))
    for s in reversed(starts):
        e = min(L0, s + K)
        v += [(RC, j) for j in range(s, e - 1)]
        v += [(LB, j) for j in range(e - 1, s - 1, -1)]
    return v + [(EB, -1)]


CASES = [(1, 1), (2, 1), (5, 1), (5, 2), (7, 3), (8, 4), (6, 6), (4, 10), (48, 1), (24, 2)]


@pytest.mark.parametrize("L,K", CASES)
@pytest.mark.parametrize("flags", [0, hms.MT_STORE_ACTS, hms.MT_NO_DOUBLE_BUFFER, hms.MT_TIE_EMBEDDINGS])
def test_visit_order_follows_block_recompute(L, K, flags):
    v = hms.plan_schedule(L, K, flags)
    assert [(x["kind"], x["layer"]) for x in v] == expected_order(L, K, bool(flags & hms.MT_STORE_ACTS))
    tied = bool(flags & hms.MT_TIE_EMBEDDINGS)
    for x in v:
        if x["kind"] in (LF, RC, LB):
            assert x["tile"] == x["layer"] + 1
        elif x["kind"] == HD:
            assert x["tile"] == (0 if tied else L + 1)
        else:
            assert x["tile"] == 0
    # recompute regenerates exactly the layers between checkpoints
    n_rc = sum(x["kind"] == RC for x in v)
    assert n_rc == (0 if flags & hms.MT_STORE_ACTS else L - (L + K - 1) // K)


@pytest.mark.parametrize("L,K", CASES)
@pytest.mark.parametrize("flags", [0, hms.MT_NO_DOUBLE_BUFFER, hms.MT_TIE_EMBEDDINGS])
def test_buffers_hold_what_each_visit_binds(L, K, flags):
    """Simulate the two device buffers: a visit without a copy finds its tile
    already there; a copy waits for the buffer's previous user; with two
    buffers the copy never targets the buffer of the visit just before it (so
    it overlaps that visit's compute)."""
    v = hms.plan_schedule(L, K, flags)
    single = bool(flags & hms.MT_NO_DOUBLE_BUFFER)
    held, last = [None, None], [-1, -1]
    prev_buf = None
    for i, x in enumerate(v):
        if x["kind"] == EB:  # the embedding gradient needs no weights on the device
            assert x["buf"] == -1 and x["h2d"] == 0
            continue
        b = x["buf"]
        assert b in ((0,) if single else (0, 1))
        assert x["buf_wait"] == last[b]
        if x["h2d"]:
            assert held[b] != x["tile"] and x["tile"] not in held[:1 if single else 2]
            if not single and prev_buf is not None:
                assert b != prev_buf
            held[b] = x["tile"]
        else:
            assert held[b] == x["tile"]
        last[b] = i
        prev_buf = b


@pytest.mark.parametrize("L", [1, 3, 48])
def test_k1_streams_every_layer_twice_and_reuses_the_last(L):
    """K = 1: each layer's weights stream in for forward and again for
    backward, except the last layer, whose backward follows the head while its
    tile is still resident; embedding and head stream once."""
    v = hms.plan_schedule(L, 1, 0)
    copies = {}
    for x in v:
        if x["h2d"]:
            copies[x["tile"]] = copies.get(x["tile"], 0) + 1
    assert copies[0] == 1 and copies[L + 1] == 1
    for i in range(1, L + 1):
        assert copies[i] == (1 if i == L else 2), i
    assert sum(copies.values()) == 2 * L + 1


def test_tied_single_layer_reuses_the_embedding_upload_for_the_head():
    v = hms.plan_schedule(1, 1, hms.MT_TIE_EMBEDDINGS)
    head = [x for x in v if x["kind"] == HD][0]
    assert head["tile"] == 0 and head["h2d"] == 0
    v2 = hms.plan_schedule(3, 1, hms.MT_TIE_EMBEDDINGS)
    assert [x for x in v2 if x["kind"] == HD][0]["h2d"] == 1  # evicted by the layers in between


@pytest.mark.parametrize("L,K", CASES)
def test_gradient_buffers_rotate(L, K):
    """Layer gradients alternate between device gradient buffers 0 and 1; the
    head and the embedding rows use buffer 2; each visit's gradients wait for
    the previous user of its buffer to have been evacuated."""
    v = hms.plan_schedule(L, K, 0)
    last = {0: -1, 1: -1, 2: -1}
    nxt = 0
    for i, x in enumerate(v):
        if x["kind"] in (EF, LF, RC):
            assert x["gbuf"] == -1
            continue
        if x["kind"] == LB:
            assert x["gbuf"] == nxt
            nxt ^= 1
        else:
            assert x["gbuf"] == 2
        assert x["gbuf_wait"] == last[x["gbuf"]]
        last[x["gbuf"]] = i


def test_bad_arguments_and_counting_call():
    lib = _lib.lib()
    assert lib.mt_plan_schedule(0, 1, 0, 0, None, 0) == _lib.MT_EINVAL
    assert lib.mt_plan_schedule(4, 0, 0, 0, None, 0) == _lib.MT_EINVAL
    assert lib.mt_plan_schedule(4, 1, -1, 0, None, 0) == _lib.MT_EINVAL
    assert lib.mt_plan_schedule(4, 1, 0, 0, None, -1) == _lib.MT_EINVAL
    assert lib.mt_plan_schedule(4, 1, 0, 0, None, 0) == len(expected_order(4, 1))


@pytest.mark.parametrize("L,K,keep", [(1, 1, 1), (5, 1, 2), (5, 2, 3), (7, 3, 2), (8, 4, 8), (8, 4, 20),
                                      (48, 1, 48), (48, 1, 30), (24, 2, 5)])
def test_kept_layers_go_backward_without_recompute(L, K, keep):
    """The last `keep` layers keep their internals: their backward visits come
    right after the head with no recompute; the rest keep the block schedule.
    keep >= L is the stored-activations schedule."""
    v = hms.plan_schedule(L, K, 0, keep)
    assert [(x["kind"], x["layer"]) for x in v] == expected_order(L, K, keep=keep)
    L0 = max(0, L - keep)
    n_rc = sum(x["kind"] == RC for x in v)
    assert n_rc == L0 - (L0 + K - 1) // K
    if keep >= L:
        assert v == hms.plan_schedule(L, K, hms.MT_STORE_ACTS)
    # every layer still has exactly one forward and one backward visit
    assert sorted(x["layer"] for x in v if x["kind"] == LB) == list(range(L))
    # the buffers hold what each visit binds (as in the block schedule)
    held = [None, None]
    for x in v:
        if x["kind"] == EB:
            continue
        if x["h2d"]:
            held[x["buf"]] = x["tile"]
        assert held[x["buf"]] == x["tile"]
