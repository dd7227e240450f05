"""Parity at the workloads' full widths, lengths and launch shapes.

(1) Per-layer parity at full shape.  One decoder layer of each workload runs
    through ``mt_layer_pass`` with that workload's whole batch x sequence,
    width, heads and ffn, so every kernel sees the launch shapes of a
    training step.  The input activations are seeded; the output gradient is
    nonzero only on the last R rows of chosen sequences.  By causality the
    oracle's tail-rows layer then gives, exactly and cheaply, x' on those
    rows, dL/dx on every row of those sequences and the layer's full weight
    gradients.  Every other sequence must receive dL/dx = 0 exactly.
(2) The attention kernels at the workloads' sequence lengths (4K with GQA,
    32K, 128K and 512K with MHA): output, log-sum-exp and dq on sampled query rows,
    dk and dv on sampled keys, each computed by the oracle one at a time.
(3) Full-width models of reduced depth against the whole oracle: loss, every
    gradient and the Adam update.  The oracle needs O(T) host work per layer
    and O(T V d) for the head in FP64, so these run at a reduced token count.
"""
import gc

import pytest
import torch

import mt_inputs
import oracle
from oracle import OracleConfig
from tests import bounds, parity

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")
from host_memory_streamed_gb300 import ops  # noqa: E402

D = torch.float64
DEV = "cuda"


def cos_rel(a, b):
    a = a.to(D).reshape(-1)
    b = b.to(D).reshape(-1)
    nb = float(b.norm())
    return float(a @ b) / max(float(a.norm()) * nb, 1e-300), float((a - b).norm()) / max(nb, 1e-300)


# ---------------------------------------------------------------------------- (1) per-layer, full shape
LAYER_CASES = {
    # workload: (tail rows R, sequences carrying the output gradient)
    "1.3b": (200, "first_last"),
    "14b": (200, "first_last"),
    "70b": (136, "first_last"),
    "7b-32k": (72, "first_last"),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_pass_full_shape_matches_oracle(name):
    s = mt_inputs.PRESETS[name].with_(n_layers=1)
    R, _ = LAYER_CASES[name]
    B, S, d = s.batch, s.seq, s.d_model
    T, t0 = B * S, S - R
    cfg = OracleConfig.from_shape(s)
    m = hms.StreamedDecoder.from_shape(s)
    try:
        lw = mt_inputs.layer_weights(s, 0, gain_jitter=0.1)
        m.load_tile(1, hms.MT_PART_W, m.pack(1, lw))
        x = mt_inputs.normal_bf16((T, d), seed=31, std=0.05)
        grad_seqs = sorted({0, B - 1})
        dy = torch.zeros(T, d, dtype=torch.bfloat16)
        for b in grad_seqs:
            dy[b * S + t0:(b + 1) * S] = mt_inputs.normal_bf16((R, d), seed=40 + b, std=1e-2)
        xd, dyd = x.to(DEV), dy.to(DEV)
        y = torch.empty(T, d, device=DEV, dtype=torch.bfloat16)
        dx = torch.full((T, d), 7.0, device=DEV, dtype=torch.bfloat16)
        m.layer_pass(0, xd, dyd, y, dx)
        torch.cuda.synchronize()
        y, dx = y.cpu(), dx.cpu()
        g_lib = m.unpack(1, m.get_tile(1, hms.MT_PART_G))
    finally:
        m.close()
    del xd, dyd
    torch.cuda.empty_cache()

    # sequences without output gradient receive none
    others = torch.ones(T, dtype=torch.bool)
    for b in grad_seqs:
        others[b * S:(b + 1) * S] = False
    assert int(torch.count_nonzero(dx[others])) == 0

    lw64 = {k: v.to(D) for k, v in lw.items()}
    cos, sin = oracle.rope_cos_sin(S, s.head_dim, s.rope_theta)
    g_ref = None
    for b in grad_seqs:
        rows = slice(b * S, (b + 1) * S)
        y_o, dx_o, g_o = oracle.layer_tail_rows(x[rows].to(D), dy[b * S + t0:(b + 1) * S].to(D), lw64, cfg, cos,
                                                sin, t0)
        c, r = cos_rel(y[b * S + t0:(b + 1) * S], y_o)
        assert c >= parity.GRAD_COS and r <= parity.GRAD_RTOL, ("x'", b, c, r)
        c, r = cos_rel(dx[rows], dx_o)
        assert c >= parity.GRAD_COS and r <= parity.GRAD_RTOL, ("dx", b, c, r)
        g_ref = g_o if g_ref is None else {k: g_ref[k] + g_o[k] for k in g_o}
        del y_o, dx_o, g_o
        gc.collect()
    bad = []
    for k in mt_inputs.LAYER_TENSORS:
        c, r = cos_rel(g_lib[k], g_ref[k])
        if not (c >= parity.GRAD_COS and r <= parity.GRAD_RTOL):
            bad.append((k, c, r))
    assert not bad, bad


# ---------------------------------------------------------------------------- (2) attention at full length
ATTN_CASES = {
    # name: (B, S, Hq, Hkv, sampled batch rows, sampled query heads, query rows, keys)
    "14b": (8, 4096, 40, 8, (0, 7), (0, 17, 39), (0, 1, 127, 128, 1000, 2049, 4094, 4095), (0, 64, 2047, 4000, 4095)),
    "7b-32k": (1, 32768, 32, 32, (0,), (0, 31), (0, 1, 4095, 16383, 16384, 32767), (32767, 32700, 32100)),
    "7b-128k": (1, 131072, 32, 32, (0,), (0, 31), (0, 127, 65536, 131071), (131071, 131000, 130900)),
    "7b-512k": (1, 524288, 32, 32, (0,), (0, 31), (0, 4095, 262144, 524287), (524287, 524200)),
}


@pytest.mark.parametrize("name", list(ATTN_CASES))
def test_attention_full_length_sampled_rows_and_keys(name):
    B, S, Hq, Hkv, bs, hs, rows, keys = ATTN_CASES[name]
    hd = 128
    T, ld = B * S, (Hq + 2 * Hkv) * hd
    qkv = mt_inputs.normal_bf16((T, ld), seed=51, std=1.4)
    do = mt_inputs.normal_bf16((T, Hq * hd), seed=52, std=1.0)
    qd, dod = qkv.to(DEV), do.to(DEV)
    o = torch.empty(T, Hq * hd, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=DEV)
    st = torch.zeros(1, device=DEV, dtype=torch.int32)
    ops.attention_fwd(qd, B, S, Hq, Hkv, hd, o, lse, st)
    dqkv = torch.zeros(T, ld, device=DEV, dtype=torch.bfloat16)
    ops.attention_bwd(qd, B, S, Hq, Hkv, hd, o, lse, dod, torch.empty(B * Hq * S, device=DEV), dqkv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o, lse, dqkv = o.cpu().to(D), lse.cpu().to(D), dqkv.cpu().to(D)
    del qd, dod
    torch.cuda.empty_cache()
    G = Hq // Hkv
    rows = list(rows)
    for b in bs:
        seq = slice(b * S, (b + 1) * S)
        x = qkv[seq]
        for h in hs:
            j = h * Hkv // Hq
            q = x[:, h * hd:(h + 1) * hd].to(D)
            k = x[:, (Hq + j) * hd:(Hq + j + 1) * hd].to(D)
            v = x[:, (Hq + Hkv + j) * hd:(Hq + Hkv + j + 1) * hd].to(D)
            o_r, lse_r, dq_r = oracle.attention_rows(q, k, v, rows, do[seq][:, h * hd:(h + 1) * hd].to(D))
            idx = [b * S + r for r in rows]
            c, r = cos_rel(o[idx, h * hd:(h + 1) * hd], o_r)
            assert r < 5e-3, (name, b, h, "o", r)
            lse_g = lse[[(b * Hq + h) * S + r for r in rows]]
            assert float((lse_g - lse_r).abs().max()) < 1e-4 * max(1.0, float(lse_r.abs().max())), (name, b, h)
            c, r = cos_rel(dqkv[idx, h * hd:(h + 1) * hd], dq_r)
            assert r < 1e-2, (name, b, h, "dq", r)
            # element-wise, each sampled row against its own bound
            do_h = do[seq][:, h * hd:(h + 1) * hd]
            rb = [bounds.attention_row(q, k, v, do_h, i) for i in rows]
            bounds.check(o[idx, h * hd:(h + 1) * hd], o_r, torch.stack([x[0] for x in rb]), f"{name} o (b{b} h{h})")
            bounds.check(dqkv[idx, h * hd:(h + 1) * hd], dq_r, torch.stack([x[1] for x in rb]),
                         f"{name} dq (b{b} h{h})")
        for j in sorted({h * Hkv // Hq for h in hs}):
            heads = range(j * G, (j + 1) * G)
            qs = torch.stack([x[:, h * hd:(h + 1) * hd] for h in heads]).to(D)
            dos = torch.stack([do[seq][:, h * hd:(h + 1) * hd] for h in heads]).to(D)
            k = x[:, (Hq + j) * hd:(Hq + j + 1) * hd].to(D)
            v = x[:, (Hq + Hkv + j) * hd:(Hq + Hkv + j + 1) * hd].to(D)
            dks, dvs, gk, gv = [], [], [], []
            for key in keys:
                dk_r, dv_r = oracle.attention_key_grads(qs, k, v, dos, key)
                dks.append(dk_r)
                dvs.append(dv_r)
                gk.append(dqkv[b * S + key, (Hq + j) * hd:(Hq + j + 1) * hd])
                gv.append(dqkv[b * S + key, (Hq + Hkv + j) * hd:(Hq + Hkv + j + 1) * hd])
                bk, bv = bounds.attention_key(qs, k, v, dos, key)
                bounds.check(gk[-1], dk_r, bk, f"{name} dk (b{b} kv{j} key {key})")
                bounds.check(gv[-1], dv_r, bv, f"{name} dv (b{b} kv{j} key {key})")
            _, r = cos_rel(torch.stack(gk), torch.stack(dks))
            assert r < 1e-2, (name, b, j, "dk", r)
            _, r = cos_rel(torch.stack(gv), torch.stack(dvs))
            assert r < 1e-2, (name, b, j, "dv", r)


# ---------------------------------------------------------------------------- (3) full width, reduced depth
MODEL_CASES = {
    "1.3b": dict(n_layers=2, ckpt_every=2, batch=2, seq=136),
    "14b": dict(n_layers=2, batch=1, seq=200),
    "70b": dict(n_layers=1, batch=1, seq=128),
    "7b-32k": dict(n_layers=2, batch=1, seq=256),
}


def _row_chunks(t, n=1 << 24):
    flat = t.reshape(-1)
    for lo in range(0, flat.numel(), n):
        yield slice(lo, min(flat.numel(), lo + n))


@pytest.mark.parametrize("name", list(MODEL_CASES))
def test_full_width_model_matches_oracle(name):
    s = mt_inputs.PRESETS[name].with_(**MODEL_CASES[name])
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    m = hms.StreamedDecoder.from_shape(s)
    try:
        m.load_weights(params)
        loss = m.train_step(tokens)
        loss_ref, grads = oracle.model_loss_and_grads(params, tokens, cfg)
        assert abs(loss - loss_ref) <= parity.LOSS_RTOL * abs(loss_ref), (loss, loss_ref)
        hcfg = parity.fp32_hyper(cfg)
        rep, ok, total = {}, 0, 0
        for i in range(m.n_tiles):
            named_g = m.unpack(i, m.get_tile(i, hms.MT_PART_G))
            named_w = m.unpack(i, m.get_tile(i, hms.MT_PART_W))
            named_m = m.unpack(i, m.get_tile(i, hms.MT_PART_M), torch.float32)
            named_v = m.unpack(i, m.get_tile(i, hms.MT_PART_V), torch.float32)
            w0 = m._tile_named(params, i)
            g0 = m._tile_named(grads, i)
            for k, g in named_g.items():
                rep[(i, k)] = cos_rel(g, g0[k])
                # Adam: reading (i) on the library's own gradient, element-wise
                # within 1 BF16 ulp; reading (ii) against the oracle's gradient
                wf, wof, gf, gof = (named_w[k].reshape(-1), w0[k].reshape(-1), g.reshape(-1), g0[k].reshape(-1))
                mf, vf = named_m[k].reshape(-1), named_v[k].reshape(-1)
                rms = float(gof.pow(2).mean().sqrt())
                for sl in _row_chunks(wf):
                    z = torch.zeros(sl.stop - sl.start, dtype=D)
                    we, me, ve = oracle.adam_update(wof[sl], gf[sl], z, z, 1, hcfg)
                    off = (wf[sl].to(D) - we).abs() > parity.adam_weight_tol(we, wof[sl])
                    if bool(off.any()):
                        ix = off.nonzero()[:6, 0]
                        raise AssertionError(
                            f"tile {i} {k}: {int(off.sum())} of {off.numel()} weights beyond 1 BF16 ulp of the "
                            f"oracle's Adam on the library's gradient; first at {(sl.start + ix).tolist()}: "
                            f"w0 {wof[sl][ix].tolist()} g {gf[sl][ix].tolist()} w_lib {wf[sl][ix].tolist()} "
                            f"w_expect {we[ix].tolist()} m_lib {mf[sl][ix].tolist()} v_lib {vf[sl][ix].tolist()}")
                    gd = gf[sl].to(D)
                    assert torch.all((mf[sl].to(D) - me).abs() <= 4 * 2.0 ** -24 * (1 - hcfg.beta1) * gd.abs())
                    assert torch.all((vf[sl].to(D) - ve).abs() <= 4 * 2.0 ** -24 * (1 - hcfg.beta2) * gd * gd)
                    wo_, _, _ = oracle.adam_update(wof[sl], oracle.round_to_bf16(gof[sl]), z, z, 1, cfg)
                    meaningful = gof[sl].abs() > 1e-3 * rms
                    total += int(meaningful.sum())
                    ok += int(((wf[sl].to(D) - wo_).abs() <= parity.bf16_ulp(wo_))[meaningful].sum())
            del named_g, named_w, named_m, named_v
            gc.collect()
        assert ok >= 0.99 * total, (ok, total)
    finally:
        m.close()
    assert all(c >= parity.GRAD_COS for c, _ in rep.values()), rep
    names = ["embed"] + [f"layer{j}" for j in range(s.n_layers)] + ["head"]
    for (i, k), (c, r) in sorted(rep.items()):
        print(f"{name} {names[i]}.{k}: cos {c:.6f} rel {r:.4f}")
    over = {key: r for key, (c, r) in rep.items() if r > parity.GRAD_RTOL}
    if over:
        # The target's normwise bound is not met for these tensors.  Reading
        # R8: BF16 tensor-core operands (the normalised activations and q/k/v
        # feeding the BF16 GEMMs and attention) force this error on any
        # implementation that stores them in BF16; the storage-precision model
        # (the same step in FP32, rounded to BF16 exactly where the library
        # stores BF16, no kernels) shows it on the same inputs.  The test
        # reports the case as an expected failure of the target, and fails
        # outright if the library's error is not that storage error (more
        # than 10 % above the model's).
        from tests import precision_model as pm
        assert s.batch == 1
        _, gm = pm.Model(pm.ALL).loss_and_grads(params, tokens, cfg)
        lines = []
        for (i, k), r in sorted(over.items()):
            tree = gm["embed"] if i == 0 else (gm["head"] if i == s.n_layers + 1 else gm["layers"][i - 1])
            _, r_model = cos_rel(tree[k], m._tile_named(grads, i)[k])
            lines.append(f"{names[i]}.{k}: library {r:.4f}, storage-precision model {r_model:.4f}")
            print(lines[-1])
            assert r <= 1.1 * r_model, (names[i], k, r, r_model)
        pytest.xfail("normwise gradient error above 2e-2 from BF16 storage of tensor-core operands: " +
                     "; ".join(lines))
