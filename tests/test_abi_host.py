"""Host-side checks of libmt.so that need no GPU: the library loads and exports
every symbol the headers declare, the CPU Adam matches the oracle, the tile
layout (queried without a handle) keeps the pages' 12-bytes-per-parameter
accounting, and bad configurations are rejected with MT_EINVAL."""
import ctypes as C
import os

import pytest
import torch

import mt_inputs
import oracle
from oracle import OracleConfig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from host_memory_streamed_gb300 import _lib, build
    build.build()
    return _lib.lib()


def test_library_exports_every_declared_symbol(lib):
    from host_memory_streamed_gb300 import _lib
    names = _lib.declared_symbols()
    assert "mt_init_model" in names and "mt_train_step" in names and "mt_op_gemm" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(shape, **kw):
    from host_memory_streamed_gb300 import _lib
    c = _lib.MtConfig()
    for k in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "batch", "seq",
              "ckpt_every", "rms_eps", "rope_theta", "lr", "beta1", "beta2", "adam_eps", "weight_decay"):
        setattr(c, k, getattr(shape, k))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("name", ["tiny", "1.3b", "14b", "70b", "7b-32k", "7b-128k"])
def test_required_device_bytes_positive_and_bounded(lib, name):
    s = mt_inputs.PRESETS[name]
    need = lib.mt_required_device_bytes(C.byref(_cfg(s)))
    assert need > 0
    # the device footprint is bounded by activations + two tile buffers, far below the model
    assert need < 280e9
    if name == "14b":
        assert need < 80e9


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(n_kv_heads=3), dict(ffn=690), dict(ckpt_every=0),
                                 dict(vocab=0), dict(batch=0), dict(seq=3, batch=1), dict(mlp_chunk_rows=100),
                                 dict(mlp_chunk_rows=128, flags=2), dict(n_experts=12, top_k=2),
                                 dict(n_experts=8, top_k=0), dict(n_experts=8, top_k=9), dict(n_experts=512, top_k=2),
                                 dict(n_experts=8, top_k=2, mlp_chunk_rows=128), dict(keep_layers=-1),
                                 dict(keep_layers=1, mlp_chunk_rows=128)])
def test_bad_config_rejected(lib, bad):
    s = mt_inputs.PRESETS["tiny"]
    assert lib.mt_required_device_bytes(C.byref(_cfg(s, **bad))) == -1
    assert lib.mt_last_error(None)


def _adam_ref(w, g, m, v, t, cfg):
    return oracle.adam_update(w, g, m, v, t, cfg)


@pytest.mark.parametrize("t", [1, 2, 7])
def test_cpu_adam_matches_oracle(lib, t):
    from tests.parity import fp32_hyper
    cfg = fp32_hyper(OracleConfig.from_shape(mt_inputs.PRESETS["tiny"]))
    gen = torch.Generator().manual_seed(10 + t)
    n = 200003
    w = (torch.randn(n, generator=gen, dtype=torch.float32) * 0.05).to(torch.bfloat16)
    g = (torch.randn(n, generator=gen, dtype=torch.float32)
         * torch.exp(torch.randn(n, generator=gen, dtype=torch.float32) * 3) * 1e-4).to(torch.bfloat16)
    g[::97] = 0.0
    m = (torch.randn(n, generator=gen, dtype=torch.float32) * 1e-5) if t > 1 else torch.zeros(n, dtype=torch.float32)
    v = (torch.rand(n, generator=gen, dtype=torch.float32) * 1e-9) if t > 1 else torch.zeros(n, dtype=torch.float32)
    wb, mb, vb = w.clone(), m.clone(), v.clone()
    rc = lib.mt_adam_host(wb.view(torch.int16).data_ptr(), g.view(torch.int16).data_ptr(), mb.data_ptr(),
                          vb.data_ptr(), n, t, cfg.lr, cfg.beta1, cfg.beta2, cfg.adam_eps, cfg.weight_decay)
    assert rc == 0
    we, me, ve = _adam_ref(w, g, m, v, t, cfg)
    diff = (wb.double() - we).abs()
    from tests.parity import adam_weight_tol
    tol = adam_weight_tol(we, w)
    assert torch.all(diff <= tol), int((diff > tol).sum())
    # FP32 moments: a few FP32 ulps of the larger term (b1 m and (1-b1) g can cancel)
    gd, md, vd = g.double(), m.double(), v.double()
    assert torch.all((mb.double() - me).abs() <= 4 * 2.0 ** -24 * (cfg.beta1 * md.abs() + (1 - cfg.beta1) * gd.abs()))
    assert torch.all((vb.double() - ve).abs() <= 4 * 2.0 ** -24 * (cfg.beta2 * vd + (1 - cfg.beta2) * gd * gd))
    # zero gradient at t = 1 leaves the weight untouched
    if t == 1:
        assert torch.equal(wb[::97], w[::97])


def test_cpu_adam_rejects_bad_step(lib):
    x = torch.zeros(4, dtype=torch.int16)
    f = torch.zeros(4, dtype=torch.float32)
    assert lib.mt_adam_host(x.data_ptr(), x.data_ptr(), f.data_ptr(), f.data_ptr(), 4, 0, 1e-4, 0.9, 0.95, 1e-8,
                            0.0) != 0


def _golden(name):
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#")[0].split()
        if line:
            vals[line[0]] = int(line[1])
    return vals


def _plan_tiles(lib, shape, **kw):
    """Every tile's layout from the library, without a handle."""
    from host_memory_streamed_gb300 import _lib
    cfg = _cfg(shape, **kw)
    n = lib.mt_plan_tile_info(C.byref(cfg), 0, None)
    assert n > 0, lib.mt_last_error(None)
    out = []
    for t in range(n):
        d = _lib.MtTileDesc()
        assert lib.mt_plan_tile_info(C.byref(cfg), t, C.byref(d)) == n
        out.append(d)
    return out


@pytest.mark.parametrize("name,kw", [("1.3b", {}), ("14b", {}), ("70b", {}), ("1.3b", {"flags": 128}),
                                     ("1.3b", {"n_experts": 8, "top_k": 2})])
def test_tile_layout_accounting(lib, name, kw):
    """The library's host tiles (queried through the C-ABI, no GPU) hold W
    (BF16) | G (BF16) | M (FP32) | V (FP32): the pages' bytes per parameter
    (tests/golden/persistent_state.txt) plus section and sub-tensor padding,
    every tensor where the layout documents it, with the parameter count of
    the architecture; tiles in the documented order (embedding, layers, head;
    no head tile when the embedding is tied)."""
    gold = _golden("persistent_state.txt")
    per_param = gold["state_bytes_per_param"]
    assert per_param == gold["weight_bytes_per_param"] + gold["grad_bytes_per_param"] + \
        gold["moment_bytes_per_param"]
    s = mt_inputs.PRESETS[name]
    tied = bool(kw.get("flags", 0) & 128)
    E = kw.get("n_experts", 0)
    tiles = _plan_tiles(lib, s, **kw)
    assert len(tiles) == s.n_layers + (1 if tied else 2)
    d, dq, dqkv = s.d_model, s.n_heads * s.head_dim, (s.n_heads + 2 * s.n_kv_heads) * s.head_dim
    if E:
        layer = [("g1", d, 0), ("wqkv", dqkv, d), ("wo", d, dq), ("g2", d, 0), ("wr", E, d),
                 ("wgu", E * 2 * s.ffn, d), ("wd", E * d, s.ffn)]
    else:
        layer = [("g1", d, 0), ("wqkv", dqkv, d), ("wo", d, dq), ("g2", d, 0), ("wgu", 2 * s.ffn, d),
                 ("wd", d, s.ffn)]
    expect = [[("E", s.vocab, d)] + ([("gf", d, 0)] if tied else [])] + [layer] * s.n_layers
    if not tied:
        expect.append([("gf", d, 0), ("wh", s.vocab, d)])
    total_params = total_bytes = 0
    for i, (t, ex) in enumerate(zip(tiles, expect)):
        assert t.kind == (0 if i == 0 else (1 if i <= s.n_layers else 2))
        assert t.n_tensors == len(ex)
        end = 0
        for k, (nm, r, c) in enumerate(ex):
            x = t.tensors[k]
            assert x.name.decode() == nm and x.ndim == (2 if c else 1)
            assert (x.shape[0], x.shape[1]) == (r, c) and x.numel == (r * c if c else r)
            assert x.offset % 256 == 0 and x.offset >= end  # 256-byte sub-tensors, in order, no overlap
            end = x.offset + 2 * x.numel
        assert t.n_params == sum(r * c if c else r for _, r, c in ex)
        # W and G: BF16 per parameter; M and V: FP32 per parameter; 4 KB sections
        assert t.w_bytes % 4096 == 0 and end <= t.w_bytes < end + 4096
        assert t.tile_bytes == 2 * t.w_bytes + 2 * (2 * t.w_bytes)  # W, G + M, V at twice the bytes
        assert per_param * t.n_params <= t.tile_bytes
        # padding: at most 255 bytes per sub-tensor plus 4 KB per W section, times six W-sized sections
        assert t.tile_bytes <= per_param * t.n_params + 6 * (256 * t.n_tensors + 4096)
        total_params += t.n_params
        total_bytes += t.tile_bytes
    if name == "14b" and not kw:
        assert tiles[1].n_params == 275261440
    if name == "70b":
        # the pages' 70B figure, at this shape's 70.55 B parameters
        assert total_params >= gold["params_70b"]
        assert total_bytes >= gold["state_bytes_70b"]
        assert total_bytes <= per_param * total_params * 1.0001


def test_plan_tile_info_rejects_bad_arguments(lib):
    from host_memory_streamed_gb300 import _lib
    s = mt_inputs.PRESETS["tiny"]
    cfg = _cfg(s)
    n = lib.mt_plan_tile_info(C.byref(cfg), 0, None)
    assert n == s.n_layers + 2
    d = _lib.MtTileDesc()
    for t in (-1, n):
        assert lib.mt_plan_tile_info(C.byref(cfg), t, C.byref(d)) == -1
        assert "tile index" in lib.mt_last_error(None).decode()
    assert lib.mt_plan_tile_info(C.byref(_cfg(s, n_heads=3, n_kv_heads=2)), 0, C.byref(d)) == -1
    assert lib.mt_plan_tile_info(None, 0, C.byref(d)) == -1


def test_header_documents_every_entry_point():
    """Every declared function has a comment block in its header."""
    from host_memory_streamed_gb300 import _lib
    txt = "".join(open(os.path.join(ROOT, "include", f)).read() for f in os.listdir(os.path.join(ROOT, "include")))
    for n in _lib.declared_symbols():
        assert n in txt


def test_cpu_adam_cancellation_within_fp32_bound(lib):
    """Where the first Adam step nearly cancels the weight (w ~ lr * |g|/(|g| + eps)),
    the host's FP32 subtraction leaves an error of a few FP32 ulps of |w|, far
    more than one BF16 ulp of the tiny result: the weight check allows the
    larger of the two (the update is computed in FP32)."""
    from tests.parity import adam_weight_tol, bf16_ulp, fp32_hyper
    cfg = fp32_hyper(OracleConfig.from_shape(mt_inputs.PRESETS["tiny"]))
    g = torch.tensor([2.9206275939941406e-06, -3.0e-6, 1e-3], dtype=torch.float32).to(torch.bfloat16)
    upd = cfg.lr * g.double().abs() / (g.double().abs() + cfg.adam_eps)
    w = (upd * g.double().sign()).to(torch.bfloat16)  # w - lr*u is then within rounding of zero
    w[2] = 0.05  # an ordinary weight
    wb, mb, vb = w.clone(), torch.zeros(3), torch.zeros(3)
    assert lib.mt_adam_host(wb.view(torch.int16).data_ptr(), g.view(torch.int16).data_ptr(), mb.data_ptr(),
                            vb.data_ptr(), 3, 1, cfg.lr, cfg.beta1, cfg.beta2, cfg.adam_eps, cfg.weight_decay) == 0
    z = torch.zeros(3, dtype=torch.float64)
    we, _, _ = oracle.adam_update(w, g, z, z, 1, cfg)
    diff = (wb.double() - we).abs()
    assert torch.all(diff <= adam_weight_tol(we, w))
    assert float(we[:2].abs().max()) < 1e-3 * float(w[:2].double().abs().min())  # the update cancels w
    assert diff[2] <= bf16_ulp(we[2:])[0]  # an ordinary weight stays within 1 BF16 ulp


def test_chunked_mlp_shrinks_the_device_arena(lib):
    """Row-chunked MLP: the [tokens, 2 ffn] activations and their gradient exist
    one chunk at a time, so the long-sequence step fits the GPU."""
    s = mt_inputs.PRESETS["7b-512k"]
    whole = lib.mt_required_device_bytes(C.byref(_cfg(s)))
    chunked = lib.mt_required_device_bytes(C.byref(_cfg(s, mlp_chunk_rows=65536)))
    assert chunked > 0 and whole - chunked > 40e9
    assert chunked < 240e9



def test_fault_injection_and_wait_probe_argument_checks(lib):
    """Both entry points validate on the host before touching a handle or the device."""
    from host_memory_streamed_gb300 import _lib
    assert lib.mt_debug_inject(None, _lib.MT_INJECT_LOADER_FAIL, 0) == _lib.MT_EINVAL
    assert lib.mt_op_wait_probe(None, 50_000_000, None) == _lib.MT_EINVAL
    for limit in (0, 999_999, 5_000_000_001):
        assert lib.mt_op_wait_probe(0x10000, limit, None) == _lib.MT_EINVAL


def test_moe_arena_grows_with_the_routed_pairs(lib):
    """MoE layers: the device arena holds the routing, the permuted rows and the
    experts' outputs of one layer pass, sized by tokens x top_k, and the same
    per-layer weight buffers as the largest tile."""
    s = mt_inputs.PRESETS["tiny"]
    dense = lib.mt_required_device_bytes(C.byref(_cfg(s)))
    k2 = lib.mt_required_device_bytes(C.byref(_cfg(s, n_experts=8, top_k=2)))
    k4 = lib.mt_required_device_bytes(C.byref(_cfg(s, n_experts=8, top_k=4)))
    assert 0 < dense < k2 < k4
    T, d, F = s.batch * s.seq, s.d_model, s.ffn
    # two more pairs per token add at least their rows of xp, yp, dyp, dxp (d each), ap (F), gup and dgup (2F)
    assert k4 - k2 >= 2 * T * (4 * d + F + 4 * F) * 2


def test_grouped_gemm_rejects_bad_arguments_before_any_launch(lib):
    """mt_op_gemm_grouped validates on the host and returns MT_EINVAL without
    touching the device (the pointers below are never dereferenced)."""
    from host_memory_streamed_gb300 import _lib
    A, B, Cp, off = 0x10000, 0x20000, 0x30000, 0x40000

    def call(layout=0, grouping=_lib.GEMM_GROUP_ROWS, offsets=off, groups=8, epi=_lib.EPI_STORE_BF16, M=1024,
             N=256, K=128, lda=128, ldb=128, ldc=256):
        return lib.mt_op_gemm_grouped(A, lda, B, ldb, M, N, K, layout, grouping, offsets, groups, epi, Cp, ldc,
                                      None, 0, None, 0, None, None)

    bad = [
        dict(groups=0), dict(groups=257), dict(offsets=None), dict(offsets=off + 2),
        dict(grouping=3), dict(layout=_lib.GEMM_A_MN),                            # rows grouping wants K-major A
        dict(epi=_lib.EPI_ROPE), dict(epi=_lib.EPI_RESIDUAL_BF16),
        dict(grouping=_lib.GEMM_GROUP_K, layout=_lib.GEMM_B_MN),                  # K grouping wants both MN-major
        dict(grouping=_lib.GEMM_GROUP_K, layout=3, epi=_lib.EPI_SWIGLU, lda=1024, ldb=256),
        dict(K=100),                                                              # K-major K not a multiple of 8
        dict(layout=4),
    ]
    for kw in bad:
        assert call(**kw) == _lib.MT_EINVAL, kw
        assert lib.mt_op_last_error()


def test_moe_padding_capacity_and_route_checks(lib):
    from host_memory_streamed_gb300 import _lib
    assert lib.mt_op_moe_rows_capacity(1000, 8, 1) == 1000
    assert lib.mt_op_moe_rows_capacity(1000, 8, 64) == 1000 + 63 * 8
    assert lib.mt_op_moe_rows_capacity(1000, 8, 0) == -1 and lib.mt_op_moe_rows_capacity(1000, 8, 257) == -1
    p = 0x10000
    for row_align in (0, 300):
        assert lib.mt_op_moe_route(p, 100, 8, 2, row_align, p, p, p, p, p, p, None) == _lib.MT_EINVAL
    assert lib.mt_op_moe_zero_pads(p, 0, 64, p, None) == _lib.MT_EINVAL


def test_rmsnorm_scratch_size_is_overflow_safe(lib):
    f = lib.mt_op_rmsnorm_bwd_scratch_floats
    assert f(130, 64) == 3 * 64 and f(128, 64) == 2 * 64 and f(0, 64) == 0
    assert f(-1, 64) == -1 and f(10, 0) == -1
    assert f((1 << 63) - 1, 1 << 20) == -1  # the product does not fit in int64
    assert f((1 << 63) - 1, 8) == ((1 << 63) - 1 + 63) // 64 * 8


def test_kept_layers_add_their_internals_to_the_arena(lib):
    """Each kept layer adds one stored set (its input and internals) to the
    device arena; keeping every layer drops the checkpoints and the shared set
    and equals MT_STORE_ACTS."""
    import host_memory_streamed_gb300 as hms
    s = mt_inputs.PRESETS["tiny"].with_(n_layers=4)
    need = [lib.mt_required_device_bytes(C.byref(_cfg(s, keep_layers=k))) for k in range(5)]
    step = need[2] - need[1]
    assert step > 0 and need[3] - need[2] == step
    assert need[4] == lib.mt_required_device_bytes(C.byref(_cfg(s, flags=hms.MT_STORE_ACTS)))
    assert lib.mt_required_device_bytes(C.byref(_cfg(s, keep_layers=9))) == need[4]


def test_binding_plans_the_tiles_without_a_gpu(lib):
    """``StreamedDecoder.plan_tiles`` returns the tiles the C-ABI describes; at
    the 14B shape they take 12 bytes per parameter plus under 0.01 % of
    padding (177 GB)."""
    import host_memory_streamed_gb300 as hms
    s = mt_inputs.PRESETS["14b"]
    tiles = hms.StreamedDecoder.plan_tiles(s)
    assert len(tiles) == s.n_layers + 2
    assert list(tiles[1]["tensors"]) == ["g1", "wqkv", "wo", "g2", "wgu", "wd"]
    assert tiles[1]["tensors"]["wgu"]["shape"] == (2 * s.ffn, s.d_model)
    params = sum(t["n_params"] for t in tiles)
    host = sum(t["tile_bytes"] for t in tiles)
    assert 12 * params <= host <= 12 * params * 1.0001
    assert 176e9 < host < 178e9
    with pytest.raises(hms.MtError):
        hms.StreamedDecoder.plan_tiles(s, n_kv_heads=7)


_ATT = dict(ldqkv=(4 + 2 * 2) * 64, batch=2, seq=100, n_heads=4, n_kv_heads=2, head_dim=64, ldo=4 * 64)


@pytest.mark.parametrize("bad,msg", [
    (dict(head_dim=96, ldqkv=8 * 96, ldo=4 * 96), "head_dim"),
    (dict(n_kv_heads=3, ldqkv=10 * 64), "multiple of n_kv_heads"),
    (dict(seq=0), "empty"),
    (dict(batch=-1), "empty"),
    (dict(ldqkv=8 * 64 - 8), "ldqkv too small"),
    (dict(ldo=4 * 64 + 4), "multiples of 8"),
    (dict(qkv=0), "null"),
    (dict(o=0x10008), "misaligned"),
    (dict(dout=0), "null dout"),
    (dict(dqkv=0x20008), "16-byte aligned"),
    (dict(rope_cos=0x30000), "cos and sin"),
])
def test_attention_ops_reject_bad_arguments_before_any_launch(lib, bad, msg):
    """The attention entry points check shapes, leading dimensions, pointers
    and alignment on the host and return MT_EINVAL with a message; nothing is
    launched (these run without a GPU; the pointers are never dereferenced)."""
    from host_memory_streamed_gb300 import _lib
    a = dict(_ATT, qkv=0x10000, o=0x20000, lse=0x30000, dout=0x40000, delta=0x50000, dqkv=0x60000,
             rope_cos=None, rope_sin=None)
    a.update(bad)
    fwd_only = {"dout", "dqkv", "rope_cos"}.isdisjoint(bad)
    if fwd_only:
        rc = lib.mt_op_attention_fwd(a["qkv"], a["ldqkv"], a["batch"], a["seq"], a["n_heads"], a["n_kv_heads"],
                                     a["head_dim"], a["o"], a["ldo"], a["lse"], None, None)
        assert rc == _lib.MT_EINVAL and msg in lib.mt_op_last_error().decode()
    rc = lib.mt_op_attention_bwd(a["qkv"], a["ldqkv"], a["batch"], a["seq"], a["n_heads"], a["n_kv_heads"],
                                 a["head_dim"], a["o"], a["ldo"], a["lse"], a["dout"], a["delta"], a["dqkv"],
                                 a["rope_cos"], a["rope_sin"], None, None)
    assert rc == _lib.MT_EINVAL and msg in lib.mt_op_last_error().decode()


A0, A1, A2, A3, A4, A5, A6 = (0x100000 * (i + 1) for i in range(7))  # 16-byte aligned stand-ins, never read
ODD = 0x100008  # 8-byte aligned only


@pytest.mark.parametrize("call,msg", [
    (lambda L: L.mt_op_rmsnorm_fwd(A0, A1, A2, A3, 10, 12, 1e-5, None), "multiple of 8"),
    (lambda L: L.mt_op_rmsnorm_fwd(A0, A1, A2, A3, -1, 64, 1e-5, None), "rows"),
    (lambda L: L.mt_op_rmsnorm_fwd(A0, A1, A2, A3, 1 << 31, 64, 1e-5, None), "rows"),
    (lambda L: L.mt_op_rmsnorm_fwd(None, A1, A2, A3, 10, 64, 1e-5, None), "null"),
    (lambda L: L.mt_op_rmsnorm_fwd(A0, A1, ODD, A3, 10, 64, 1e-5, None), "16-byte"),
    (lambda L: L.mt_op_rmsnorm_bwd(A0, A1, A2, A3, None, A4, A5, None, 10, 64, None), "null"),
    (lambda L: L.mt_op_rmsnorm_bwd(A0, A1, A2, A3, None, A4, None, A6, 0, 64, None), "null"),
    (lambda L: L.mt_op_rmsnorm_bwd(A0, A1, A2, A3, ODD, A4, A5, A6, 10, 64, None), "16-byte"),
    (lambda L: L.mt_op_rmsnorm_bwd_noalloc(A0, A1, A2, None, None, A4, A5, 10, 64, None), "null"),
    (lambda L: L.mt_op_rmsnorm_bwd_noalloc(ODD, A1, A2, A3, None, A4, A5, 10, 64, None), "16-byte"),
    (lambda L: L.mt_op_swiglu_bwd(A0, A1, A2, -1, 16, None), "rows"),
    (lambda L: L.mt_op_swiglu_bwd(A0, None, A2, 4, 16, None), "null"),
    (lambda L: L.mt_op_swiglu_bwd(A0, A1, ODD, 4, 16, None), "16-byte"),
    (lambda L: L.mt_op_transpose(A0, 4, 10, 9, A1, 4, None), "leading dimension"),
    (lambda L: L.mt_op_transpose(A0, 4, 10, 10, A1, 3, None), "leading dimension"),
    (lambda L: L.mt_op_transpose(None, 4, 10, 10, A1, 4, None), "null"),
    (lambda L: L.mt_op_cross_entropy(A0, 4, 0, A1, 0.25, A2, A3, None, None), "vocab"),
    (lambda L: L.mt_op_cross_entropy(A0, 4, 64, None, 0.25, A2, A3, None, None), "null"),
    (lambda L: L.mt_op_cross_entropy(ODD, 4, 64, A1, 0.25, A2, A3, None, None), "16-byte"),
    (lambda L: L.mt_op_embedding_fwd(A0, A1, A2, 5, 60, 100, None, None), "multiple of 8"),
    (lambda L: L.mt_op_embedding_fwd(A0, A1, A2, 5, 64, 0, None, None), "V positive"),
    (lambda L: L.mt_op_embedding_fwd(A0, None, A2, 5, 64, 100, None, None), "null"),
    (lambda L: L.mt_op_embedding_fwd(A0, ODD, A2, 5, 64, 100, None, None), "16-byte"),
    (lambda L: L.mt_op_embedding_bwd(A0, None, A2, A3, 100, 64, None), "null"),
    (lambda L: L.mt_op_embedding_bwd(A0, A1, A2, ODD, 100, 64, None), "16-byte"),
    (lambda L: L.mt_op_gemm(None, 64, A1, 64, 256, 256, 64, 0, A2, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "null A or B"),
    (lambda L: L.mt_op_gemm(A0, 64, A1, 64, 256, 256, 64, 0, ODD, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "C not 16-byte"),
    (lambda L: L.mt_op_gemm(A0, 64, A1, 64, 0, 256, 64, 0, A2, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "positive"),
    (lambda L: L.mt_op_gemm(A0, 60, A1, 64, 256, 256, 60, 0, A2, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "multiple of 8"),
    (lambda L: L.mt_op_gemm(A0, 64, A1, 64, 256, 256, 64, 1, A2, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "residual"),
    (lambda L: L.mt_op_gemm(A0, 64, A1, 64, 256, 256, 64, 5, A2, 256, None, 0, None, 0, None, None, 256, 128, 64,
                            None, None), "RoPE tables"),
    (lambda L: L.mt_op_gemm(A0, 64, A1, 64, 256, 256, 64, 9, A2, 256, None, 0, None, 0, None, None, 0, 0, 0,
                            None, None), "unknown epilogue"),
    (lambda L: L.mt_op_moe_gather(A0, 64, None, 2, 10, 64, A2, None), "null"),
    (lambda L: L.mt_op_moe_gather(ODD, 64, A1, 2, 10, 64, A2, None), "16-byte"),
    (lambda L: L.mt_op_moe_zero_pads(A0, 10, 64, ODD, None), "16-byte"),
    (lambda L: L.mt_op_moe_combine(A0, None, A2, 5, 2, 64, None, A4, None), "null"),
    (lambda L: L.mt_op_moe_combine_bwd(A0, A1, A2, A3, 5, 2, 64, A5, None, None), "null"),
    (lambda L: L.mt_op_moe_gate_bwd(A0, A1, None, 5, 8, 2, A4, None), "null"),
    (lambda L: L.mt_op_moe_scatter_bwd(A0, A1, 5, 2, 64, None, None, None), "null"),
])
def test_elementwise_ops_reject_bad_arguments_before_any_launch(lib, call, msg):
    """Each per-kernel entry point checks sizes, pointers and the alignment
    its 16-byte vector accesses need on the host, returning MT_EINVAL with a
    message (no launch: these run without a GPU and the pointers are never
    dereferenced)."""
    from host_memory_streamed_gb300 import _lib
    assert call(lib) == _lib.MT_EINVAL
    assert msg in lib.mt_op_last_error().decode()
