"""ctypes loader of libmt.so and the prototypes of its C-ABI (include/mt.h, include/mt_ops.h).

The product path has no fallback: if the library is missing this raises.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmt.so")

MT_OK, MT_EINVAL, MT_ENOMEM, MT_ECUDA, MT_ETIMEDOUT, MT_ESTATE, MT_ENONFINITE, MT_EINTERNAL = 0, -1, -2, -3, -4, -5, -6, -7
ERROR_NAMES = {0: "MT_OK", -1: "MT_EINVAL", -2: "MT_ENOMEM", -3: "MT_ECUDA", -4: "MT_ETIMEDOUT",
               -5: "MT_ESTATE", -6: "MT_ENONFINITE", -7: "MT_EINTERNAL"}

MT_RESIDENT, MT_STORE_ACTS, MT_NO_DOUBLE_BUFFER, MT_DEBUG_CHECKS, MT_TIME_KERNELS, MT_TRACE, MT_VISIT_LOG, \
    MT_TIE_EMBEDDINGS, MT_ASYNC_ADAM, MT_DIRECT_GRADS, MT_DIRECT_WEIGHTS = 1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024
MT_PART_W, MT_PART_G, MT_PART_M, MT_PART_V = 0, 1, 2, 3

EPI_STORE_BF16, EPI_RESIDUAL_BF16, EPI_F32, EPI_F32_ACCUMULATE, EPI_SWIGLU, EPI_ROPE, EPI_SWIGLU_BWD = range(7)
GEMM_A_MN, GEMM_B_MN = 1, 2  # operand layouts of mt_op_gemm_layout
GEMM_GROUP_ROWS, GEMM_GROUP_K = 1, 2  # groupings of mt_op_gemm_grouped


class MtConfig(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
        ("head_dim", C.c_int32), ("ffn", C.c_int32), ("vocab", C.c_int32),
        ("rms_eps", C.c_float), ("rope_theta", C.c_float),
        ("batch", C.c_int32), ("seq", C.c_int32), ("ckpt_every", C.c_int32),
        ("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("adam_eps", C.c_float),
        ("weight_decay", C.c_float),
        ("n_adam_threads", C.c_int32), ("n_pack_threads", C.c_int32), ("n_grad_slabs", C.c_int32),
        ("grad_slab_bytes", C.c_int64), ("stage_bytes", C.c_int64), ("timeout_ms", C.c_int64),
        ("flags", C.c_uint32), ("mlp_chunk_rows", C.c_int64), ("n_experts", C.c_int32), ("top_k", C.c_int32),
        ("keep_layers", C.c_int32), ("replica_rank", C.c_int32), ("n_replicas", C.c_int32),
        ("replica_name", C.c_char * 48),
    ]


class MtTensorDesc(C.Structure):
    _fields_ = [("name", C.c_char * 16), ("ndim", C.c_int32), ("shape", C.c_int64 * 2),
                ("offset", C.c_int64), ("numel", C.c_int64)]


class MtTileDesc(C.Structure):
    _fields_ = [("kind", C.c_int32), ("n_tensors", C.c_int32), ("n_params", C.c_int64),
                ("w_bytes", C.c_int64), ("tile_bytes", C.c_int64), ("tensors", MtTensorDesc * 8)]


class MtInterval(C.Structure):
    _fields_ = [("kind", C.c_int32), ("visit", C.c_int32), ("t0_ms", C.c_double), ("t1_ms", C.c_double)]


SPAN_COMPUTE, SPAN_H2D, SPAN_D2H = 0, 1, 2


class MtVisit(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("kind", "tile", "layer", "buf", "h2d", "buf_wait", "gbuf", "gbuf_wait")]


# host-side fault injection (mt_debug_inject) and the device wait probe's status code
(MT_INJECT_NONE, MT_INJECT_LOADER_FAIL, MT_INJECT_D2H_FAIL, MT_INJECT_ACCUM_FAIL, MT_INJECT_ADAM_FAIL,
 MT_INJECT_LOADER_STALL) = range(6)
MT_STATUS_WAIT_PROBE = 7

VISIT_EMBED_FWD, VISIT_LAYER_FWD, VISIT_HEAD, VISIT_RECOMPUTE, VISIT_LAYER_BWD, VISIT_EMBED_BWD = range(6)


class MtStepStats(C.Structure):
    _fields_ = [
        ("loss", C.c_double), ("step_ms", C.c_double), ("gpu_compute_ms", C.c_double),
        ("h2d_ms", C.c_double), ("d2h_ms", C.c_double), ("wait_weights_ms", C.c_double),
        ("adam_ms", C.c_double), ("adam_tail_ms", C.c_double), ("gemm_ms", C.c_double),
        ("gemm_flops", C.c_double), ("gemm_launches", C.c_int64), ("kernel_launches", C.c_int64),
        ("h2d_bytes", C.c_int64), ("d2h_bytes", C.c_int64), ("flops_executed", C.c_int64),
        ("flops_model", C.c_int64), ("arena_high_water", C.c_int64), ("step", C.c_int64),
        ("visit_gap_ms", C.c_double), ("host_pre_ms", C.c_double), ("tail_grads_ms", C.c_double),
        ("tail_adam_ms", C.c_double), ("tail_rest_ms", C.c_double),
    ]


_lib = None


def lib():
    """Load libmt.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with host_memory_streamed_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
    fp = C.POINTER(C.c_float)
    sig = {
        "mt_required_device_bytes": (i64, [C.POINTER(MtConfig)]),
        "mt_init_model": (C.c_int, [C.POINTER(MtConfig), vp, sz, vp, vp, vp, C.POINTER(vp)]),
        "mt_plan_schedule": (i32, [i32, i32, i32, C.c_uint32, C.POINTER(MtVisit), i32]),
        "mt_debug_inject": (C.c_int, [vp, i32, i32]),
        "mt_op_wait_probe": (C.c_int, [vp, i64, vp]),
        "mt_tile_count": (C.c_int, [vp]),
        "mt_tile_info": (C.c_int, [vp, C.c_int, C.POINTER(MtTileDesc)]),
        "mt_plan_tile_info": (C.c_int, [C.POINTER(MtConfig), C.c_int, C.POINTER(MtTileDesc)]),
        "mt_load_layer_tile": (C.c_int, [vp, C.c_int, C.c_int, vp, sz]),
        "mt_train_step": (C.c_int, [vp, vp, sz, fp]),
        "mt_train_step_device_tokens": (C.c_int, [vp, vp, sz, fp]),
        "mt_layer_pass": (C.c_int, [vp, i32, vp, vp, vp, vp]),
        "mt_train_step_micro": (C.c_int, [vp, vp, sz, i32, fp]),
        "mt_train_step_grads": (C.c_int, [vp, vp, sz, fp]),
        "mt_apply_adam": (C.c_int, [vp]),
        "mt_get_layer_tile": (C.c_int, [vp, C.c_int, C.c_int, vp, sz]),
        "mt_get_step_stats": (C.c_int, [vp, C.POINTER(MtStepStats)]),
        "mt_get_step": (i64, [vp]),
        "mt_set_step": (C.c_int, [vp, i64]),
        "mt_replica_barrier": (C.c_int, [vp]),
        "mt_sync": (C.c_int, [vp]),
        "mt_get_timeline": (i64, [vp, C.POINTER(MtInterval), i64]),
        "mt_last_error": (C.c_char_p, [vp]),
        "mt_free": (None, [vp]),
        "mt_adam_host": (C.c_int, [vp, vp, vp, vp, sz, i64, f32, f32, f32, f32, f32]),
        "mt_op_last_error": (C.c_char_p, []),
        "mt_op_gemm": (C.c_int, [vp, i64, vp, i64, i32, i32, i32, i32, vp, i64, vp, i64, vp, i64,
                                 vp, vp, i32, i32, i32, vp, vp]),
        "mt_op_gemm_layout": (C.c_int, [vp, i64, vp, i64, i32, i32, i32, i32, i32, vp, i64, vp, i64, vp, vp]),
        "mt_op_attention_fwd": (C.c_int, [vp, i64, i32, i32, i32, i32, i32, vp, i64, vp, vp, vp]),
        "mt_op_attention_bwd": (C.c_int, [vp, i64, i32, i32, i32, i32, i32, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]),
        "mt_op_rmsnorm_fwd": (C.c_int, [vp, vp, vp, vp, i64, i32, f32, vp]),
        "mt_op_rmsnorm_bwd_scratch_floats": (i64, [i64, i32]),
        "mt_op_rmsnorm_bwd": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, vp]),
        "mt_op_swiglu_bwd": (C.c_int, [vp, vp, vp, i64, i32, vp]),
        "mt_op_transpose": (C.c_int, [vp, i64, i64, i64, vp, i64, vp]),
        "mt_op_cross_entropy": (C.c_int, [vp, i64, i32, vp, f32, vp, vp, vp, vp]),
        "mt_op_embedding_fwd": (C.c_int, [vp, vp, vp, i64, i32, i32, vp, vp]),
        "mt_op_embedding_bwd": (C.c_int, [vp, vp, vp, vp, i32, i32, vp]),
        "mt_op_gemm_grouped": (C.c_int, [vp, i64, vp, i64, i32, i32, i32, i32, i32, vp, i32, i32, vp, i64, vp, i64,
                                         vp, i64, vp, vp]),
        "mt_op_moe_sort_scratch_ints": (i64, [i64, i32]),
        "mt_op_moe_rows_capacity": (i64, [i64, i32, i32]),
        "mt_op_moe_route": (C.c_int, [vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
        "mt_op_moe_zero_pads": (C.c_int, [vp, i64, i32, vp, vp]),
        "mt_op_moe_gather": (C.c_int, [vp, i64, vp, i32, i64, i32, vp, vp]),
        "mt_op_moe_combine": (C.c_int, [vp, vp, vp, i64, i32, i32, vp, vp, vp]),
        "mt_op_moe_combine_bwd": (C.c_int, [vp, vp, vp, vp, i64, i32, i32, vp, vp, vp]),
        "mt_op_moe_gate_bwd": (C.c_int, [vp, vp, vp, i64, i32, i32, vp, vp]),
        "mt_op_moe_scatter_bwd": (C.c_int, [vp, vp, i64, i32, i32, vp, vp, vp]),
        "mt_op_flag_nonfinite": (C.c_int, [vp, i64, vp, vp]),
        "mt_op_rmsnorm_bwd_noalloc": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, i64, i32, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name, None)
        if f is None:
            continue
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def declared_symbols():
    """Every function name declared in include/*.h (parsed from the headers)."""
    import re
    inc = os.path.join(os.path.dirname(HERE), "include")
    names = []
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            txt = open(os.path.join(inc, fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(mt_\w+)\s*\(", txt)
    return sorted(set(names))
