"""GB300-native layer-streamed decoder training step (MegaTrain's hot path).

Thin Python binding over ``libmt.so`` (C-ABI in ``include/mt.h`` and
``include/mt_ops.h``): argument marshalling only.  Every step of the training
path runs in the library's CUDA kernels and C++ runtime; PyTorch provides the
device arena and the three CUDA streams.  There is no CPU fallback: if the
library is missing or no GPU is present, constructing a model raises.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import (MT_ASYNC_ADAM, MT_DEBUG_CHECKS, MT_DIRECT_GRADS, MT_DIRECT_WEIGHTS, MT_NO_DOUBLE_BUFFER, MT_PART_G, MT_PART_M, MT_PART_V,
                   MT_PART_W, MT_RESIDENT, MT_STORE_ACTS, MT_TIE_EMBEDDINGS, MT_TIME_KERNELS, MT_TRACE, MT_VISIT_LOG,
                   ERROR_NAMES)

__all__ = ["StreamedDecoder", "MtError", "ops", "plan_schedule", "MT_RESIDENT", "MT_STORE_ACTS", "MT_NO_DOUBLE_BUFFER",
           "MT_DEBUG_CHECKS", "MT_TIME_KERNELS", "MT_TRACE", "MT_VISIT_LOG", "MT_TIE_EMBEDDINGS", "MT_PART_W",
           "MT_PART_G", "MT_PART_M", "MT_PART_V", "MT_ASYNC_ADAM", "MT_DIRECT_GRADS", "MT_DIRECT_WEIGHTS"]

LAYER_NAMES = ("g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")


def plan_schedule(n_layers: int, ckpt_every: int = 1, flags: int = 0, keep_layers: int = 0) -> list[dict]:
    """The visit order of one training step (``mt_plan_schedule``): a list of
    dicts with kind, tile, layer, buf, h2d, buf_wait, gbuf, gbuf_wait.  Host
    only; needs no GPU."""
    lib = _lib.lib()
    n = lib.mt_plan_schedule(n_layers, ckpt_every, keep_layers, flags, None, 0)
    if n < 0:
        raise MtError(n, "mt_plan_schedule: bad arguments")
    out = (_lib.MtVisit * n)()
    lib.mt_plan_schedule(n_layers, ckpt_every, keep_layers, flags, out, n)
    return [{f: getattr(v, f) for f, _ in _lib.MtVisit._fields_} for v in out]


def _tile_dict(d) -> dict:
    """An ``mt_tile_desc`` as a dict: kind, n_params, w_bytes, tile_bytes and
    the tensors by name (shape, byte offset in the W section, numel)."""
    tensors = {}
    for k in range(d.n_tensors):
        t = d.tensors[k]
        shape = (t.shape[0], t.shape[1]) if t.ndim == 2 else (t.shape[0],)
        tensors[t.name.decode()] = dict(shape=shape, offset=t.offset, numel=t.numel)
    return dict(kind=d.kind, n_params=d.n_params, w_bytes=d.w_bytes, tile_bytes=d.tile_bytes, tensors=tensors)


class MtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _bf16_bytes(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.uint8).reshape(-1)


class StreamedDecoder:
    """One model handle: host tiles, device arena, three streams, worker threads."""

    def __init__(self, n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab, batch, seq, *,
                 ckpt_every=1, rms_eps=1e-5, rope_theta=1e4, lr=1e-4, beta1=0.9, beta2=0.95, adam_eps=1e-8,
                 weight_decay=0.0, n_adam_threads=0, n_pack_threads=0, n_grad_slabs=0, grad_slab_bytes=0,
                 stage_bytes=0, timeout_ms=0, flags=0, mlp_chunk_rows=0, n_experts=0, top_k=0, keep_layers=0,
                 replica_group=None, device=None):
        """keep_layers: how many of the last layers keep their internals on the
        device from forward to backward (no recompute for them); "auto" keeps as
        many as fit in the device's free memory (less ``KEEP_MARGIN``).

        replica_group: ``(name, rank, n)`` makes this handle replica ``rank`` of
        ``n`` data-parallel replicas of one model whose host tiles live once, in
        the shared-memory segment ``name`` (see ``replicas``)."""
        if not torch.cuda.is_available():
            raise RuntimeError("a CUDA device is required (the library has no CPU path)")
        self._L = _lib.lib()
        cfg = _lib.MtConfig()
        for k, v in dict(n_layers=n_layers, d_model=d_model, n_heads=n_heads, n_kv_heads=n_kv_heads,
                         head_dim=head_dim, ffn=ffn, vocab=vocab, rms_eps=rms_eps, rope_theta=rope_theta,
                         batch=batch, seq=seq, ckpt_every=ckpt_every, lr=lr, beta1=beta1, beta2=beta2,
                         adam_eps=adam_eps, weight_decay=weight_decay, n_adam_threads=n_adam_threads,
                         n_pack_threads=n_pack_threads, n_grad_slabs=n_grad_slabs,
                         grad_slab_bytes=grad_slab_bytes, stage_bytes=stage_bytes, timeout_ms=timeout_ms,
                         flags=flags, mlp_chunk_rows=mlp_chunk_rows, n_experts=n_experts, top_k=top_k).items():
            setattr(cfg, k, v)
        if replica_group is not None:
            name, rank, n = replica_group
            cfg.replica_name, cfg.replica_rank, cfg.n_replicas = name.encode(), int(rank), int(n)
        self.cfg = cfg
        self.device = torch.device(device or "cuda")
        cfg.keep_layers = self.fit_keep_layers(cfg, self.device) if keep_layers == "auto" else int(keep_layers)
        self.keep_layers = min(int(cfg.keep_layers), n_layers)
        need = self._L.mt_required_device_bytes(C.byref(cfg))
        if need < 0:
            raise MtError(need, self._L.mt_last_error(None).decode())
        self.arena_bytes = int(need)
        self.arena = torch.empty(self.arena_bytes, dtype=torch.uint8, device=self.device)
        self.streams = [torch.cuda.Stream(self.device) for _ in range(3)]
        h = C.c_void_p()
        rc = self._L.mt_init_model(C.byref(cfg), self.arena.data_ptr(), self.arena_bytes,
                                   *(s.cuda_stream for s in self.streams), C.byref(h))
        if rc != 0:
            raise MtError(rc, self._L.mt_last_error(None).decode())
        self._h = h
        self.n_tiles = self._L.mt_tile_count(h)
        self.infos = [self.tile_info(i) for i in range(self.n_tiles)]
        # tied embeddings: tile 0 holds E and gf, and there is no head tile
        self.tied = bool(flags & MT_TIE_EMBEDDINGS)

    KEEP_MARGIN = 6 << 30  # device bytes left free when keep_layers is "auto"

    @classmethod
    def fit_keep_layers(cls, cfg, device) -> int:
        """The most layers whose internals fit, with the rest of the arena, in
        the device's free memory less KEEP_MARGIN (0 when none does)."""
        torch.cuda.empty_cache()  # blocks torch caches count as used
        free, _ = torch.cuda.mem_get_info(device)
        budget = free - cls.KEEP_MARGIN
        lib = _lib.lib()

        def need(k):
            c = _lib.MtConfig.from_buffer_copy(cfg)
            c.keep_layers = k
            n = lib.mt_required_device_bytes(C.byref(c))
            if n < 0:
                raise MtError(n, lib.mt_last_error(None).decode())
            return n
        lo, hi = 0, int(cfg.n_layers)
        if need(hi) <= budget:  # every layer kept also drops the checkpoints and block buffers
            return hi
        if need(0) > budget:
            return 0
        while lo < hi:  # largest k with need(k) <= budget (need grows with k)
            mid = (lo + hi + 1) // 2
            if need(mid) <= budget:
                lo = mid
            else:
                hi = mid - 1
        return lo

    @staticmethod
    def _shape_cfg(s, kw):
        cfg = _lib.MtConfig()
        for k in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "batch", "seq",
                  "ckpt_every", "rms_eps", "rope_theta", "lr", "beta1", "beta2", "adam_eps", "weight_decay"):
            setattr(cfg, k, getattr(s, k))
        for k, v in kw.items():
            setattr(cfg, k, v)
        return cfg

    @staticmethod
    def required_device_bytes(s, **kw) -> int:
        """Device arena bytes a model of shape ``s`` (and the given options) needs."""
        cfg = StreamedDecoder._shape_cfg(s, kw)
        need = _lib.lib().mt_required_device_bytes(C.byref(cfg))
        if need < 0:
            raise MtError(need, _lib.lib().mt_last_error(None).decode())
        return int(need)

    @staticmethod
    def plan_tiles(s, **kw) -> list[dict]:
        """The host tiles a model of shape ``s`` (and the given options) will
        have, as ``tile_info`` describes them, without a handle or a GPU
        (``mt_plan_tile_info``); their ``tile_bytes`` sum to the host memory
        the tile store takes."""
        cfg = StreamedDecoder._shape_cfg(s, kw)
        lib = _lib.lib()
        n = lib.mt_plan_tile_info(C.byref(cfg), 0, None)
        if n < 0:
            raise MtError(n, lib.mt_last_error(None).decode())
        out = []
        for i in range(n):
            d = _lib.MtTileDesc()
            rc = lib.mt_plan_tile_info(C.byref(cfg), i, C.byref(d))
            if rc < 0:
                raise MtError(rc, lib.mt_last_error(None).decode())
            out.append(_tile_dict(d))
        return out

    @classmethod
    def from_shape(cls, s, **kw):
        kw.setdefault("n_experts", getattr(s, "n_experts", 0))
        kw.setdefault("top_k", getattr(s, "top_k", 0))
        return cls(s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, s.ffn, s.vocab, s.batch, s.seq,
                   ckpt_every=s.ckpt_every, rms_eps=s.rms_eps, rope_theta=s.rope_theta, lr=s.lr, beta1=s.beta1,
                   beta2=s.beta2, adam_eps=s.adam_eps, weight_decay=s.weight_decay, **kw)

    # ------------------------------------------------------------------ plumbing
    def _check(self, rc):
        if rc != 0:
            raise MtError(rc, self._L.mt_last_error(self._h).decode())

    def debug_inject(self, what: int, visit: int = 0):
        """Arm a host-side failure for the next step (``mt_debug_inject``):
        one of the ``_lib.MT_INJECT_*`` kinds at the first visit >= ``visit``."""
        rc = self._L.mt_debug_inject(self._h, what, visit)
        if rc != 0:
            raise MtError(rc, "mt_debug_inject: bad arguments")

    def close(self):
        if getattr(self, "_h", None):
            for s in self.streams:
                s.synchronize()
            self._L.mt_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def tile_info(self, i):
        d = _lib.MtTileDesc()
        self._check(self._L.mt_tile_info(self._h, i, C.byref(d)))
        return _tile_dict(d)

    def _part_bytes(self, i, part):
        w = self.infos[i]["w_bytes"]
        return w if part in (MT_PART_W, MT_PART_G) else 2 * w

    def load_tile(self, i, part, buf: torch.Tensor):
        buf = buf.contiguous()
        assert buf.device.type == "cpu" and buf.numel() * buf.element_size() == self._part_bytes(i, part)
        self._check(self._L.mt_load_layer_tile(self._h, i, part, buf.data_ptr(), self._part_bytes(i, part)))

    def get_tile(self, i, part) -> torch.Tensor:
        out = torch.empty(self._part_bytes(i, part), dtype=torch.uint8)
        self._check(self._L.mt_get_layer_tile(self._h, i, part, out.data_ptr(), out.numel()))
        return out

    # ------------------------------------------------------------------ named <-> tile layout
    def _named_to_slots(self, i, named):
        kind = self.infos[i]["kind"]
        if kind == 0:
            return {"E": named["E"], "gf": named["gf"]} if self.tied else {"E": named["E"]}
        if kind == 2:
            return {"gf": named["gf"], "wh": named["wh"]}
        if "experts" in named:  # MoE layer: experts stacked, each expert's gate/up rows interleaved
            ex = named["experts"]
            wgu = torch.cat([torch.stack([e["wg"], e["wu"]], dim=1).reshape(-1, e["wg"].shape[1]) for e in ex], 0)
            return {"g1": named["g1"], "wqkv": torch.cat([named["wq"], named["wk"], named["wv"]], 0),
                    "wo": named["wo"], "g2": named["g2"], "wr": named["wr"], "wgu": wgu,
                    "wd": torch.cat([e["wd"] for e in ex], 0)}
        wgu = torch.stack([named["wg"], named["wu"]], dim=1).reshape(-1, named["wg"].shape[1])
        return {"g1": named["g1"], "wqkv": torch.cat([named["wq"], named["wk"], named["wv"]], 0),
                "wo": named["wo"], "g2": named["g2"], "wgu": wgu, "wd": named["wd"]}

    def _slots_to_named(self, i, slots):
        kind = self.infos[i]["kind"]
        if kind != 1:
            return slots
        c = self.cfg
        q, kv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
        wqkv, wgu = slots["wqkv"], slots["wgu"]
        if "wr" in slots:
            E, F, d = c.n_experts, c.ffn, c.d_model
            wgu = wgu.reshape(E, 2 * F, -1)
            wd = slots["wd"].reshape(E, d, F)
            return {"g1": slots["g1"], "wq": wqkv[:q], "wk": wqkv[q:q + kv], "wv": wqkv[q + kv:],
                    "wo": slots["wo"], "g2": slots["g2"], "wr": slots["wr"],
                    "experts": [{"wg": wgu[e, 0::2], "wu": wgu[e, 1::2], "wd": wd[e]} for e in range(E)]}
        return {"g1": slots["g1"], "wq": wqkv[:q], "wk": wqkv[q:q + kv], "wv": wqkv[q + kv:],
                "wo": slots["wo"], "g2": slots["g2"], "wg": wgu[0::2], "wu": wgu[1::2], "wd": slots["wd"]}

    def pack(self, i, named, dtype=torch.bfloat16) -> torch.Tensor:
        """Named tensors of tile i -> the tile section bytes (W/G for BF16, M/V for FP32)."""
        slots = self._named_to_slots(i, named)
        esz = 2 if dtype == torch.bfloat16 else 4
        out = torch.zeros(self.infos[i]["w_bytes"] * esz // 2, dtype=torch.uint8)
        for name, meta in self.infos[i]["tensors"].items():
            t = slots[name].to(dtype).contiguous().reshape(-1)
            assert t.numel() == meta["numel"], (name, t.numel(), meta["numel"])
            o = meta["offset"] * esz // 2
            out[o:o + meta["numel"] * esz] = t.view(torch.uint8)
        return out

    def unpack(self, i, raw: torch.Tensor, dtype=torch.bfloat16):
        esz = 2 if dtype == torch.bfloat16 else 4
        slots = {}
        for name, meta in self.infos[i]["tensors"].items():
            o = meta["offset"] * esz // 2
            slots[name] = raw[o:o + meta["numel"] * esz].view(dtype).reshape(meta["shape"]).clone()
        return self._slots_to_named(i, slots)

    def _tile_named(self, params, i):
        if i == 0:
            return dict(params["embed"], gf=params["head"]["gf"]) if self.tied else params["embed"]
        if i == self.n_tiles - 1 and not self.tied:
            return params["head"]
        return params["layers"][i - 1]

    def load_weights(self, params):
        """params: {'embed': {'E'}, 'layers': [{g1,wq,...}], 'head': {'gf','wh'}} of BF16 tensors
        ('head': {'gf'} alone with tied embeddings)."""
        for i in range(self.n_tiles):
            self.load_tile(i, MT_PART_W, self.pack(i, self._tile_named(params, i)))

    def _collect(self, part, dtype):
        out = {"embed": None, "layers": [], "head": None}
        for i in range(self.n_tiles):
            named = self.unpack(i, self.get_tile(i, part), dtype)
            if i == 0:
                if self.tied:
                    out["head"] = {"gf": named.pop("gf")}
                out["embed"] = named
            elif i == self.n_tiles - 1 and not self.tied:
                out["head"] = named
            else:
                out["layers"].append(named)
        return out

    def weights(self):
        return self._collect(MT_PART_W, torch.bfloat16)

    def grads(self):
        return self._collect(MT_PART_G, torch.bfloat16)

    def moments(self):
        return self._collect(MT_PART_M, torch.float32), self._collect(MT_PART_V, torch.float32)

    # ------------------------------------------------------------------ the step
    def train_step(self, tokens: torch.Tensor) -> float:
        """tokens: int32 [B, S+1] on the host (or on the GPU). Returns the loss."""
        loss = C.c_float()
        tok = tokens.to(torch.int32).contiguous()
        if tok.is_cuda:
            rc = self._L.mt_train_step_device_tokens(self._h, tok.data_ptr(), tok.numel(), C.byref(loss))
        else:
            rc = self._L.mt_train_step(self._h, tok.data_ptr(), tok.numel(), C.byref(loss))
        self._check(rc)
        return loss.value

    def train_step_micro(self, tokens: torch.Tensor) -> float:
        """tokens: int32 [n_micro, B, S+1] on the host; one step with gradient
        accumulation over the n_micro micro-batches.  Returns the mean loss."""
        tok = tokens.to(torch.int32).contiguous()
        if tok.dim() != 3 or tok.is_cuda:
            raise TypeError("tokens must be a host tensor [n_micro, batch, seq + 1]")
        loss = C.c_float()
        self._check(self._L.mt_train_step_micro(self._h, tok.data_ptr(), tok.numel(), tok.shape[0], C.byref(loss)))
        return loss.value

    def train_step_grads(self, tokens: torch.Tensor) -> float:
        """Forward and backward of one step without the optimizer: the tiles'
        G sections receive the gradient of the mean loss over these tokens
        (host int32 [B, S+1]); weights, moments and the step are unchanged.
        Returns the loss.  See ``apply_adam``."""
        loss = C.c_float()
        tok = tokens.to(torch.int32).contiguous()
        if tok.is_cuda:
            raise TypeError("tokens must be a host tensor [batch, seq + 1]")
        self._check(self._L.mt_train_step_grads(self._h, tok.data_ptr(), tok.numel(), C.byref(loss)))
        return loss.value

    def apply_adam(self):
        """One Adam step of every tile from its G section as it stands; advances the step."""
        self._check(self._L.mt_apply_adam(self._h))

    def layer_pass(self, layer, x_in, dx_out=None, x_out=None, dx_in=None):
        """One decoder layer's forward (and backward, given dx_out) on device BF16
        [batch*seq, d_model] activations; the layer's gradient lands in its host
        tile's G section (see ``grads``).  Adam does not run."""
        c = self.cfg
        shape = (c.batch * c.seq, c.d_model)
        for t, n in ((x_in, "x_in"), (dx_out, "dx_out"), (x_out, "x_out"), (dx_in, "dx_in")):
            if t is None:
                continue
            if not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != shape or not t.is_contiguous():
                raise TypeError(f"{n} must be a contiguous CUDA bfloat16 tensor of shape {shape}")
        p = lambda t: None if t is None else t.data_ptr()
        torch.cuda.current_stream(self.device).synchronize()
        self._check(self._L.mt_layer_pass(self._h, int(layer), p(x_in), p(dx_out), p(x_out), p(dx_in)))

    def timeline(self) -> list[tuple[int, int, float, float]]:
        """(kind, visit, t0_ms, t1_ms) spans of the last step (``mt_get_timeline``;
        MT_TIME_KERNELS): compute per visit, H2D and D2H per chunk copy."""
        n = self._L.mt_get_timeline(self._h, None, 0)
        if n < 0:
            raise MtError(int(n), "mt_get_timeline failed")
        out = (_lib.MtInterval * max(1, n))()
        n = self._L.mt_get_timeline(self._h, out, n)
        return [(out[i].kind, out[i].visit, out[i].t0_ms, out[i].t1_ms) for i in range(n)]

    def sync(self):
        """Wait for every pending Adam update (``mt_sync``; MT_ASYNC_ADAM)."""
        self._check(self._L.mt_sync(self._h))

    def barrier(self):
        """Replica group: wait until every replica has called ``barrier`` as
        often as this one (``mt_replica_barrier``); no-op outside a group."""
        self._check(self._L.mt_replica_barrier(self._h))

    def stats(self) -> dict:
        st = _lib.MtStepStats()
        self._check(self._L.mt_get_step_stats(self._h, C.byref(st)))
        return {k: getattr(st, k) for k, _ in st._fields_}

    @property
    def step(self) -> int:
        return int(self._L.mt_get_step(self._h))

    @step.setter
    def step(self, v):
        self._check(self._L.mt_set_step(self._h, int(v)))


def adam_host(w_bits: torch.Tensor, g_bits: torch.Tensor, m: torch.Tensor, v: torch.Tensor, t: int, lr: float,
              beta1: float, beta2: float, eps: float, weight_decay: float = 0.0):
    """The library's CPU Adam (in place) on BF16 w/g (as int16 bit views) and FP32 m/v."""
    L = _lib.lib()
    rc = L.mt_adam_host(w_bits.data_ptr(), g_bits.data_ptr(), m.data_ptr(), v.data_ptr(), w_bits.numel(), t,
                        lr, beta1, beta2, eps, weight_decay)
    if rc != 0:
        raise MtError(rc, "mt_adam_host rejected its arguments")


from . import ops  # noqa: E402
