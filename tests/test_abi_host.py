"""Host-side checks of libmt.so that need no GPU: the library loads and exports
every symbol the headers declare, the CPU Adam matches the oracle, the tile
layout keeps the 12-bytes-per-parameter accounting, and bad configurations are
rejected with MT_EINVAL."""
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


def test_tile_layout_accounting():
    """Layer tiles hold W (BF16) | G (BF16) | M (FP32) | V (FP32), each section
    page aligned: 12 bytes per parameter plus padding (the pages' 12P
    accounting, 70B -> at least 840 GB)."""
    for name in ("1.3b", "14b", "70b"):
        s = mt_inputs.PRESETS[name]
        shapes = mt_inputs.layer_tensor_shapes(s)
        n = sum(int(torch.tensor(v).prod()) for v in shapes.values())
        per_layer = 12 * n
        total = s.n_layers * per_layer + 12 * (2 * s.vocab * s.d_model + s.d_model)
        if name == "70b":
            assert total >= 840e9
        if name == "14b":
            assert abs(n - 275261440) == 0


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
