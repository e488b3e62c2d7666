"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
AssertionError on a mismatch. They check the oracle against closed forms,
invariants of the routing, brute force on tiny inputs (every expert applied to
every token, then masked), library routines (numpy / scipy / torch CPU in fp64)
and values printed on the pages (``tests/golden``). ``test_oracle_pins.py``
runs them on the normal build; ``test_oracle_plants.py`` runs them on builds
with a deliberate mistake compiled in and requires that some pin fails.
"""
from __future__ import annotations

import json
import math
import os
from types import SimpleNamespace

import numpy as np
import scipy.special
import torch
import torch.nn.functional as Fn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def wl(**kw):
    base = dict(n_tokens=8, d_model=8, d_ff=16, n_experts=4, top_k=2, capacity_factor=0.0,
                gating="softmax_topk", act="gelu", dtype="f32", has_bias=False, n_shared=0,
                d_ff_shared=0, aux_alpha=0.01)
    base.update(kw)
    return SimpleNamespace(**base)


def rand_layer(w, seed, scale_router=1.0):
    """fp32 numpy tensors for a layer described by ``w`` (tiny sizes only)."""
    rs = np.random.RandomState(seed)
    N, d, F, E, S, Fs = w.n_tokens, w.d_model, w.d_ff, w.n_experts, w.n_shared, w.d_ff_shared
    f = lambda *s: rs.standard_normal(s).astype(np.float32)
    t = dict(x=f(N, d), w_router=(f(E, d) * scale_router).astype(np.float32), logit_bias=None,
             w1=f(E, F, d) / np.float32(math.sqrt(d)), w2=f(E, d, F) / np.float32(math.sqrt(F)))
    t["w3"] = f(E, F, d) / np.float32(math.sqrt(d)) if w.act == "swiglu" else None
    t["b1"] = f(E, F) * np.float32(0.1) if w.has_bias else None
    t["b2"] = f(E, d) * np.float32(0.1) if w.has_bias else None
    if S:
        t["ws1"] = f(S, Fs, d) / np.float32(math.sqrt(d))
        t["ws3"] = f(S, Fs, d) / np.float32(math.sqrt(d)) if w.act == "swiglu" else None
        t["ws2"] = f(S, d, Fs) / np.float32(math.sqrt(Fs))
        t["bs1"] = f(S, Fs) * np.float32(0.1) if w.has_bias else None
        t["bs2"] = f(S, d) * np.float32(0.1) if w.has_bias else None
    return {k: (None if v is None else np.ascontiguousarray(v, np.float32)) for k, v in t.items()}


# --- library-routine restatements used by the brute-force checks -------------
def torch_expert(t, e, x64, act, has_bias, shared=False):
    """One expert on rows x64 [n, d] with torch CPU fp64 library ops (F.linear, F.gelu, F.silu)."""
    pre = "ws" if shared else "w"
    bpre = "bs" if shared else "b"
    W1 = torch.from_numpy(t[pre + "1"][e].astype(np.float64))
    W2 = torch.from_numpy(t[pre + "2"][e].astype(np.float64))
    xt = torch.from_numpy(x64)
    if act == "gelu":
        b1 = torch.from_numpy(t[bpre + "1"][e].astype(np.float64)) if has_bias else None
        b2 = torch.from_numpy(t[bpre + "2"][e].astype(np.float64)) if has_bias else None
        return Fn.linear(Fn.gelu(Fn.linear(xt, W1, b1)), W2, b2).numpy()
    W3 = torch.from_numpy(t[pre + "3"][e].astype(np.float64))
    return Fn.linear(Fn.silu(Fn.linear(xt, W1)) * Fn.linear(xt, W3), W2).numpy()


def brute_force_layer(w, t, logits):
    """Every expert on every token, then masked: the layer by its defining formula.

    Top-k by a stable lexicographic sort, gates by scipy softmax, dropping by the
    pages' own "nonzero in token order, keep the first C" formulation.
    """
    N, E, k = w.n_tokens, w.n_experts, w.top_k
    x64 = t["x"].astype(np.float64)
    L = logits.astype(np.float64)
    dense = np.stack([torch_expert(t, e, x64, w.act, w.has_bias) for e in range(E)], axis=1)  # [N,E,d]
    p = scipy.special.softmax(L, axis=1)
    weight = np.zeros((N, E))
    if w.gating == "expert_choice":
        C = min(N, math.ceil(N * k * (w.capacity_factor if w.capacity_factor > 0 else 1.0) / E))
        keys = p.astype(np.float32)  # selection keys: the fp32 softmax-over-experts probabilities
        for e in range(E):
            order = np.lexsort((np.arange(N), -keys[:, e].astype(np.float64)))
            for tok in order[:C]:
                weight[tok, e] = p[tok, e]
    else:
        order = np.lexsort((np.tile(np.arange(E), (N, 1)), -L), axis=1)[:, :k]  # desc value, asc index
        if w.gating == "topk_softmax":
            sel = np.take_along_axis(L, order, 1)
            gsel = scipy.special.softmax(sel, axis=1)
        else:
            gsel = np.take_along_axis(p, order, 1)
            if w.gating == "softmax_topk_renorm":
                gsel = gsel / gsel.sum(1, keepdims=True)
        C = math.ceil(N * k * w.capacity_factor / E) if w.capacity_factor > 0 else N
        choice = order
        for e in range(E):
            mask = (choice == e)
            index = np.nonzero(mask.any(axis=1))[0][:C]
            for tok in index:
                weight[tok, e] = gsel[tok][mask[tok]][0]
    out = np.einsum("ne,ned->nd", weight, dense)
    for s in range(w.n_shared):
        out += torch_expert(t, s, x64, w.act, w.has_bias, shared=True)
    return out


# --- pins -------------------------------------------------------------------
def pin_capacity(o):
    """C = ceil(N*k*cf/E), no limit for cf <= 0 (hand-computed values)."""
    cases = [  # (N, k, cf, E, C)
        (64, 2, 1.25, 8, 20), (8192, 2, 1.25, 8, 2560), (8192, 6, 1.25, 160, 384),
        (10, 1, 1.25, 8, 2), (16384, 8, 1.0, 256, 512), (100, 3, 0.0, 7, 100), (4, 4, 1.25, 2, 4),
    ]
    for N, k, cf, E, C in cases:
        cfg = o.config(wl(n_tokens=N, top_k=min(k, E), n_experts=E, capacity_factor=cf), top_k=k)
        assert o.capacity(cfg) == C, (N, k, cf, E, o.capacity(cfg), C)


def pin_router_logits(o):
    """Router logits equal numpy's fp64 matmul rounded to fp32 (within 1 ulp)."""
    w = wl(n_tokens=13, d_model=24, n_experts=5)
    t = rand_layer(w, 1)
    t["logit_bias"] = np.linspace(0, 2, 5).astype(np.float32)
    cfg = o.config(w)
    L = o.router_logits(cfg, t["x"], o.weights(t))
    ref = (t["x"].astype(np.float64) @ t["w_router"].astype(np.float64).T + t["logit_bias"]).astype(np.float32)
    assert np.all(np.abs(L - ref) <= np.spacing(np.abs(ref))), np.max(np.abs(L - ref))


def pin_softmax(o):
    """Softmax and log-sum-exp equal scipy's."""
    rs = np.random.RandomState(2)
    L = (rs.standard_normal((9, 11)) * 5).astype(np.float32)
    p, lse = o.softmax(L)
    np.testing.assert_allclose(p, scipy.special.softmax(L.astype(np.float64), axis=1), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(L.astype(np.float64), axis=1), rtol=1e-13)


def pin_topk(o):
    """Top-k by value descending, equal values to the lower expert index."""
    L = np.array([[1, 3, 3, 2], [0, 0, 0, 0], [5, -1, 5, 5], [-2, -1, -3, -1]], np.float32)
    assert o.topk(L, 2).tolist() == [[1, 2], [0, 1], [0, 2], [1, 3]]
    assert o.topk(L, 4).tolist() == [[1, 2, 3, 0], [0, 1, 2, 3], [0, 2, 3, 1], [1, 3, 0, 2]]
    rs = np.random.RandomState(3)
    L = rs.randint(-3, 3, size=(50, 7)).astype(np.float32)  # many ties
    for k in (1, 3, 7):
        ref = np.lexsort((np.tile(np.arange(7), (50, 1)), -L), axis=1)[:, :k]
        assert np.array_equal(o.topk(L, k), ref)


def pin_gates(o):
    """Gate variants: A = p[idx]; A' and B sum to 1 and agree; a two-expert closed form."""
    rs = np.random.RandomState(4)
    N, E, k = 20, 6, 3
    L = (rs.standard_normal((N, E)) * 2).astype(np.float32)
    idx = o.topk(L, k)
    gA = o.gates(o.config(wl(n_tokens=N, n_experts=E, top_k=k, gating="softmax_topk")), L, idx)
    gR = o.gates(o.config(wl(n_tokens=N, n_experts=E, top_k=k, gating="softmax_topk_renorm")), L, idx)
    gB = o.gates(o.config(wl(n_tokens=N, n_experts=E, top_k=k, gating="topk_softmax")), L, idx)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(gA, np.take_along_axis(p, idx, 1), rtol=1e-13)
    np.testing.assert_allclose(gR.sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(gB.sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(gR, gB, rtol=1e-12)
    assert np.all(gA.sum(1) < 1.0)
    # logits (0, ln 3): top-2 order (1, 0), renormalised gates (3/4, 1/4); A gives the same here (k = E)
    L2 = np.array([[0.0, math.log(3.0)]], np.float32)
    i2 = o.topk(L2, 2)
    assert i2.tolist() == [[1, 0]]
    for g in ("softmax_topk", "softmax_topk_renorm", "topk_softmax"):
        gg = o.gates(o.config(wl(n_tokens=1, n_experts=2, top_k=2, gating=g)), L2, i2)
        np.testing.assert_allclose(gg[0], [0.75, 0.25], rtol=1e-7)


def _check_assign_invariants(idx, a, C, E):
    N, k = idx.shape
    row_of, off, counts, kept = a["row_of"], a["expert_off"], a["counts"], a["kept"]
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert np.all(kept == np.minimum(counts, C))
    assert off[0] == 0 and np.array_equal(np.diff(off), kept)
    R = int(off[-1])
    assert R == N * k - a["dropped"]
    rows = row_of[row_of >= 0]
    assert np.array_equal(np.sort(rows), np.arange(R))  # bijection onto kept (t, j)
    for e in range(E):
        ts, js = np.nonzero((idx == e) & (row_of >= 0))
        r = row_of[ts, js]
        assert np.all((r >= off[e]) & (r < off[e + 1]))
        assert np.all(np.diff(r) > 0) and np.all(np.diff(ts) > 0)  # token order inside the segment


def pin_assign(o):
    """Dropping keeps each expert's first C tokens in token order (the pages' nonzero()[:C])."""
    rs = np.random.RandomState(5)
    for N, E, k, cf in [(40, 4, 2, 1.0), (64, 8, 2, 1.25), (33, 5, 3, 0.6), (16, 6, 6, 1.25), (25, 3, 1, 0.0)]:
        L = (rs.standard_normal((N, E)) + np.linspace(0, 2, E)).astype(np.float32)
        idx = o.topk(L, k)
        cfg = o.config(wl(n_tokens=N, n_experts=E, top_k=k, capacity_factor=cf))
        C = o.capacity(cfg)
        a = o.assign(cfg, idx, C)
        _check_assign_invariants(idx, a, C, E)
        for e in range(E):
            mask = idx == e
            index = np.nonzero(mask.any(axis=1))[0]
            kept_tokens = set(index[:C].tolist())
            got = set(np.nonzero(((idx == e) & (a["row_of"] >= 0)).any(axis=1))[0].tolist())
            assert got == kept_tokens


def pin_zero_router(o):
    """W_r = 0: all logits tie, every token picks experts 0..k-1; closed-form gates and stats."""
    N, E, k, cf = 40, 8, 2, 1.25
    w = wl(n_tokens=N, d_model=8, n_experts=E, top_k=k, capacity_factor=cf)
    t = rand_layer(w, 6)
    t["w_router"][:] = 0
    C = math.ceil(N * k * cf / E)  # 13
    for gating, gexp in (("softmax_topk", 1.0 / E), ("softmax_topk_renorm", 1.0 / k), ("topk_softmax", 1.0 / k)):
        cfg = o.config(w, gating=__import__("oracle").GATING[gating])
        r = o.route(cfg, t["x"], o.weights(t))
        assert np.all(r["idx"] == np.arange(k))
        np.testing.assert_allclose(r["gate"], gexp, rtol=1e-14)
        assert r["kept"].tolist() == [min(N, C)] * k + [0] * (E - k)
        assert np.all(r["row_of"][C:] == -1) and np.all(r["row_of"][:C] >= 0)
        assert r["dropped"] == k * (N - C)
        st = r["stats"]
        np.testing.assert_allclose(st["P"], 1.0 / E, rtol=1e-14)
        np.testing.assert_allclose(st["aux_loss"], 0.01, rtol=1e-13)  # alpha exactly, whatever f is
        np.testing.assert_allclose(st["z_loss"], math.log(E) ** 2, rtol=1e-13)
        np.testing.assert_allclose(st["mean_lse_sq"], math.log(E) ** 2, rtol=1e-13)
        np.testing.assert_allclose(st["f"], [0.5, 0.5] + [0.0] * (E - 2), rtol=1e-14)
    cfg = o.config(w, gating=3, capacity_factor=1.0)
    r = o.route(cfg, t["x"], o.weights(t))
    C_ec = math.ceil(N * k / E)
    assert np.array_equal(r["sel"], np.tile(np.arange(C_ec), (E, 1)))  # ties -> lowest token ids


def pin_uniform_usage(o):
    """Cyclic routing makes f uniform, so aux = alpha * sum P = alpha for any P."""
    N, E, k = 32, 8, 2
    L = np.zeros((N, E), np.float32)
    for t_ in range(N):
        for j in range(k):
            L[t_, (t_ * k + j) % E] = 5.0 - j
    L += (np.random.RandomState(7).standard_normal((N, E)) * 0.1).astype(np.float32)
    cfg = o.config(wl(n_tokens=N, n_experts=E, top_k=k))
    r = o.route(cfg, None, None, logits=L)
    np.testing.assert_allclose(r["stats"]["f"], 1.0 / E, rtol=1e-14)
    np.testing.assert_allclose(r["stats"]["aux_loss"], 0.01, rtol=1e-12)
    # the loss grows when usage concentrates: all tokens on one expert pair
    L2 = np.zeros((N, E), np.float32)
    L2[:, 0], L2[:, 1] = 3.0, 2.0
    r2 = o.route(cfg, None, None, logits=L2)
    assert r2["stats"]["aux_loss"] > 0.01


def pin_stats_formula(o):
    """f, P, aux, z against scipy on random logits (library routines)."""
    rs = np.random.RandomState(8)
    N, E, k = 30, 6, 2
    L = (rs.standard_normal((N, E)) * 3).astype(np.float32)
    cfg = o.config(wl(n_tokens=N, n_experts=E, top_k=k, aux_alpha=0.02))
    r = o.route(cfg, None, None, logits=L)
    L64 = L.astype(np.float64)
    P = scipy.special.softmax(L64, axis=1).mean(0)
    onehot = np.zeros((N, k, E))
    np.put_along_axis(onehot, r["idx"][:, :, None].astype(np.int64), 1.0, axis=2)
    f = onehot.mean(axis=(0, 1))
    np.testing.assert_allclose(r["stats"]["P"], P, rtol=1e-12)
    np.testing.assert_allclose(r["stats"]["f"], f, rtol=1e-14)
    np.testing.assert_allclose(r["stats"]["aux_loss"], 0.02 * E * (f * P).sum(), rtol=1e-12)
    lse = scipy.special.logsumexp(L64, axis=1)
    np.testing.assert_allclose(r["stats"]["z_loss"], lse.mean() ** 2, rtol=1e-12)
    np.testing.assert_allclose(r["stats"]["mean_lse_sq"], (lse ** 2).mean(), rtol=1e-12)


def pin_single_expert_is_dense_ffn(o):
    """E = 1, k = 1, no cap: the layer is one dense FFN with gate 1 (torch F.linear/gelu/silu, fp64)."""
    for act, bias in (("gelu", True), ("gelu", False), ("swiglu", False)):
        w = wl(n_tokens=7, d_model=12, d_ff=20, n_experts=1, top_k=1, act=act, has_bias=bias)
        t = rand_layer(w, 9)
        cfg = o.config(w)
        ow = o.weights(t)
        r = o.route(cfg, t["x"], ow)
        out = o.outputs(cfg, t["x"], ow, r)
        ref = torch_expert(t, 0, t["x"].astype(np.float64), act, bias)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def pin_activation_zero(o):
    """gelu(0) = silu(0) = 0: with x = 0 a GELU expert returns b2 and a SwiGLU expert 0."""
    w = wl(n_tokens=1, d_model=8, d_ff=16, n_experts=2, top_k=1, act="gelu", has_bias=True)
    t = rand_layer(w, 10)
    t["b1"][:] = 0
    ow = o.weights(t)
    y = o.expert_apply(o.config(w), ow, 1, np.zeros(8))
    np.testing.assert_array_equal(y, t["b2"][1].astype(np.float64))
    w2 = wl(n_tokens=1, d_model=8, d_ff=16, n_experts=2, top_k=1, act="swiglu")
    t2 = rand_layer(w2, 11)
    y2 = o.expert_apply(o.config(w2), o.weights(t2), 0, np.zeros(8))
    np.testing.assert_array_equal(y2, 0.0)


def pin_brute_force(o):
    """Sparse dispatch equals dense-then-mask on tiny layers, every gating, k = 1..E, with and without drops."""
    case = 0
    for gating in ("softmax_topk", "softmax_topk_renorm", "topk_softmax", "expert_choice"):
        for act, bias in (("gelu", True), ("swiglu", False)):
            for E in (1, 3, 6):
                for k in sorted({1, 2, E}):
                    if k > E:
                        continue
                    for cf in ((0.0, 1.0) if gating != "expert_choice" else (1.0, 0.5)):
                        case += 1
                        N = 5 + (case * 7) % 12
                        w = wl(n_tokens=N, d_model=8, d_ff=12, n_experts=E, top_k=k, gating=gating,
                               act=act, has_bias=bias, capacity_factor=cf,
                               n_shared=case % 3 == 0 and 1 or 0, d_ff_shared=8)
                        t = rand_layer(w, 100 + case, scale_router=2.0)
                        cfg = o.config(w)
                        ow = o.weights(t)
                        r = o.route(cfg, t["x"], ow)
                        out = o.outputs(cfg, t["x"], ow, r)
                        ref = brute_force_layer(w, t, r["logits"])
                        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12, err_msg=str(w))


def pin_dense_softmax_mixture(o):
    """k = E, no cap, gating A: the layer is the softmax-weighted sum of every expert."""
    w = wl(n_tokens=9, d_model=8, d_ff=12, n_experts=5, top_k=5)
    t = rand_layer(w, 12, scale_router=2.0)
    cfg = o.config(w)
    ow = o.weights(t)
    r = o.route(cfg, t["x"], ow)
    out = o.outputs(cfg, t["x"], ow, r)
    x64 = t["x"].astype(np.float64)
    p = scipy.special.softmax(r["logits"].astype(np.float64), axis=1)
    ref = sum(p[:, e:e + 1] * torch_expert(t, e, x64, "gelu", False) for e in range(5))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def pin_expert_choice(o):
    """Expert choice: exactly C tokens per expert, the top-C by key (ties to lower t), ascending."""
    rs = np.random.RandomState(13)
    N, E, k = 37, 5, 2
    keys = rs.randint(0, 6, size=(N, E)).astype(np.float32)  # many ties
    cfg = o.config(wl(n_tokens=N, n_experts=E, top_k=k, gating="expert_choice", capacity_factor=1.0))
    C = o.capacity(cfg)
    assert C == math.ceil(N * k / E)
    sel = o.expert_choice(cfg, keys, C)
    for e in range(E):
        ref = np.sort(np.lexsort((np.arange(N), -keys[:, e]))[:C])
        assert np.array_equal(sel[e], ref)
    L = rs.standard_normal((N, E)).astype(np.float32)
    r = o.route(cfg, None, None, logits=L)
    np.testing.assert_allclose(r["stats"]["f"], 1.0 / E, rtol=1e-14)
    np.testing.assert_allclose(r["stats"]["aux_loss"], 0.01, rtol=1e-12)  # alpha * sum P


def pin_bf16_inputs_and_mimic(o):
    """bf16 storage widens exactly; mimic rounding gives bf16 values close to the exact output."""
    w = wl(n_tokens=6, d_model=16, d_ff=32, n_experts=3, top_k=2, dtype="bf16", act="swiglu")
    t32 = rand_layer(w, 14)
    tb = {k: (None if v is None else torch.from_numpy(v).to(torch.bfloat16)) for k, v in t32.items()}
    as_u16 = {k: (None if v is None else v.view(torch.int16).numpy().view(np.uint16)) for k, v in tb.items()}
    as_f32 = {k: (None if v is None else v.float().numpy()) for k, v in tb.items()}
    cfg_b = o.config(w)
    cfg_f = o.config(w, dtype=0)
    rb = o.route(cfg_b, as_u16["x"], o.weights(as_u16))
    rf = o.route(cfg_f, as_f32["x"], o.weights(as_f32))
    assert np.array_equal(rb["logits"], rf["logits"])
    ob = o.outputs(cfg_b, as_u16["x"], o.weights(as_u16), rb)
    of = o.outputs(cfg_f, as_f32["x"], o.weights(as_f32), rf)
    np.testing.assert_array_equal(ob, of)
    cfg_m = o.config(w, mimic_bf16=1)
    om = o.outputs(cfg_m, as_u16["x"], o.weights(as_u16), rb)
    assert np.array_equal(om, torch.from_numpy(om).float().to(torch.bfloat16).double().numpy())
    rms = np.sqrt((of ** 2).mean())
    assert np.max(np.abs(om - of)) <= 2e-2 * rms


def pin_page_entropy(o):
    """The collapse-detector entropies the aigrafen.se page prints."""
    g = json.load(open(os.path.join(GOLDEN, "routing_entropy.json")))
    for case in g["cases"]:
        assert round(o.entropy(case["distribution"]), 3) == case["entropy"], case
    assert round(math.log(8), 3) == g["maximum"]


def pin_passthrough(o):
    """Dropped-token pass-through: a token with no kept expert outputs its own input
    (plus the shared experts) exactly; a token with at least one kept expert is not
    affected. Logits are set by hand so the drop pattern is known."""
    N, E, k = 6, 3, 2
    L = np.zeros((N, E), np.float32)
    L[:, 0] = 5.0                 # every token's first choice: expert 0
    L[:3, 1] = 1.0                # tokens 0-2 then expert 1, tokens 3-5 expert 2
    L[3:, 2] = 1.0
    for shared in (0, 1):
        w = wl(n_tokens=N, d_model=8, d_ff=12, n_experts=E, top_k=k, capacity_factor=0.5,
               n_shared=shared, d_ff_shared=8)
        t = rand_layer(w, 21)
        cfg_off = o.config(w)
        cfg_on = o.config(w, passthrough=1)
        assert o.capacity(cfg_off) == 2
        ow = o.weights(t)
        r = o.route(cfg_off, None, None, logits=L)
        # expert 0 keeps tokens 0, 1; expert 1 keeps 0, 1 (drops 2); expert 2 keeps 3, 4 (drops 5)
        kept_any = (r["row_of"] >= 0).any(axis=1)
        assert kept_any.tolist() == [True, True, False, True, True, False]
        off = o.outputs(cfg_off, t["x"], ow, r)
        on = o.outputs(cfg_on, t["x"], ow, r)
        x64 = t["x"].astype(np.float64)
        np.testing.assert_array_equal(on[kept_any], off[kept_any])
        np.testing.assert_array_equal(on[~kept_any], off[~kept_any] + x64[~kept_any])
        if not shared:
            np.testing.assert_array_equal(off[~kept_any], 0.0)
            np.testing.assert_array_equal(on[~kept_any], x64[~kept_any])
    # expert choice: a token picked by no expert passes through
    w = wl(n_tokens=8, d_model=8, d_ff=12, n_experts=2, top_k=1, gating="expert_choice", capacity_factor=0.5)
    t = rand_layer(w, 22)
    Lec = np.zeros((8, 2), np.float32)
    Lec[:, 0] = np.arange(8, dtype=np.float32)   # expert 0 prefers late tokens, expert 1 early ones
    r = o.route(o.config(w), None, None, logits=Lec)
    picked = np.zeros(8, bool)
    picked[r["sel"].ravel()] = True
    assert picked.sum() < 8
    on = o.outputs(o.config(w, passthrough=1), t["x"], o.weights(t), r)
    np.testing.assert_array_equal(on[~picked], t["x"].astype(np.float64)[~picked])


def pin_assign_shard(o):
    """Capacity over a batch cut into contiguous shards: each shard assigns its tokens
    with the earlier shards' per-expert counts as rank base, and the kept pairs and
    their ranks equal the unsharded assignment; base = 0 is the unsharded rule."""
    rs = np.random.RandomState(23)
    for N, E, k, cf, cuts in [(60, 4, 2, 1.0, (20, 45)), (96, 8, 3, 0.75, (32, 64)), (50, 5, 1, 1.25, (1, 49)),
                              (40, 6, 2, 0.0, (17,))]:
        L = (rs.standard_normal((N, E)) + np.linspace(0, 2, E)).astype(np.float32)
        idx = o.topk(L, k)
        cfg = o.config(wl(n_tokens=N, n_experts=E, top_k=k, capacity_factor=cf))
        C = o.capacity(cfg)
        full = o.assign(cfg, idx, C)
        zero = o.assign_shard(cfg, idx, C, np.zeros(E, np.int32))
        for key in ("row_of", "expert_off", "counts", "kept", "dropped"):
            assert np.array_equal(np.asarray(zero[key]), np.asarray(full[key])), key
        # global (expert, rank) of every kept pair, unsharded
        ref = {}
        for tt, jj in zip(*np.nonzero(full["row_of"] >= 0)):
            e = int(idx[tt, jj])
            ref[(int(tt), int(jj))] = (e, int(full["row_of"][tt, jj] - full["expert_off"][e]))
        bounds = (0,) + tuple(cuts) + (N,)
        base = np.zeros(E, np.int32)
        got, kept, dropped = {}, np.zeros(E, np.int64), 0
        for a, b in zip(bounds[:-1], bounds[1:]):
            cfg_s = o.config(wl(n_tokens=b - a, n_experts=E, top_k=k, capacity_factor=cf))
            sh = o.assign_shard(cfg_s, np.ascontiguousarray(idx[a:b]), C, base)
            _check_shard_rows(sh, E)
            for tt, jj in zip(*np.nonzero(sh["row_of"] >= 0)):
                e = int(idx[a + tt, jj])
                got[(int(a + tt), int(jj))] = (e, int(base[e] + sh["row_of"][tt, jj] - sh["expert_off"][e]))
            kept += sh["kept"]
            dropped += sh["dropped"]
            base = base + sh["counts"]
        assert got == ref
        assert np.array_equal(kept, full["kept"]) and dropped == full["dropped"]
        assert np.array_equal(base, full["counts"])


def _check_shard_rows(sh, E):
    """A shard's rows are a bijection onto [0, rows), expert-contiguous."""
    rows = sh["row_of"][sh["row_of"] >= 0]
    assert np.array_equal(np.sort(rows), np.arange(int(sh["expert_off"][-1])))
    assert np.array_equal(np.diff(sh["expert_off"]), sh["kept"])


def pin_round_bf16_nearest_even(o):
    """The mimic mode's bf16 rounding is round-to-nearest-even: torch's bf16 cast (a
    library routine) on random values, exact halfway cases and their neighbours."""
    rs = np.random.RandomState(31)
    vals = list((rs.standard_normal(2000) * np.exp2(rs.randint(-30, 30, 2000))).astype(np.float32))
    for m in (0x3F80, 0x3F81, 0x4049, 0xC2AB, 0x0080):  # bf16 patterns: 1.0, 1+2^-7, ~3.14, negative, tiny normal
        base = np.uint32(m) << 16
        for low in (0x7FFF, 0x8000, 0x8001):  # just below, exactly at and just above the halfway point
            vals.append(np.array([base | low], np.uint32).view(np.float32)[0])
    vals = np.array(vals, np.float32)
    got = np.array([o.round_bf16(v) for v in vals], np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(got, ref)


def pin_mxfp8_dequant(o):
    """E4M3 code values against the format's closed forms and torch's float8_e4m3fn
    conversion (a library routine); MX scales are powers of two per 32 elements."""
    import oracle as orc
    v = orc.e4m3_value(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0xFE] == -448.0 and v[0x3C] == 1.5
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.sum(np.isnan(v)) == 2
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ok = ~np.isnan(v)
    np.testing.assert_array_equal(v[ok], lib[ok])
    codes = np.array([[0x38] * 32 + [0x3C] * 32], np.uint8)
    scales = np.array([[127 + 3, 127 - 2]], np.uint8)
    np.testing.assert_array_equal(orc.mxfp8_dequant(codes, scales), [[8.0] * 32 + [1.5 / 4] * 32])


def _e4m3_nearest_code(y):
    """Brute force: the E4M3 code (0..126) whose value is nearest to each y >= 0, ties
    to the even code, values above 448 to 448 (the saturating conversion)."""
    import oracle as orc
    mags = orc.e4m3_value(np.arange(127, dtype=np.uint8))
    y = np.asarray(y, np.float64)
    dist = np.abs(y[:, None] - mags[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equally near codes take the even one (two candidates at most)
    even = cand & (np.arange(127)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return np.where(y >= 448.0, 126, code).astype(np.uint8)


def pin_e4m3_rounding(o):
    """MXFP8 element rounding: nearest E4M3 value, ties to the even code, saturating at
    448, against brute force over the code table and torch's float8_e4m3fn cast (a
    library routine) below 448. A block led by 300 has scale 2^0, so its other elements'
    codes are the plain E4M3 roundings."""
    import oracle as orc
    mags = orc.e4m3_value(np.arange(127, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2
    rs = np.random.RandomState(41)
    ys = np.concatenate([mids, mids * (1 + 2.0 ** -40), mids * (1 - 2.0 ** -40), mags,
                         rs.uniform(0, 448, 600), np.exp2(rs.uniform(-12, 8.8, 600)),
                         [448.0, 449.0, 463.9, 464.0, 470.0, 500.0, 0.0, 2.0 ** -10, 3 * 2.0 ** -11]])
    ys = ys[: (len(ys) // 31) * 31].reshape(-1, 31)
    blocks = np.concatenate([np.full((len(ys), 1), 300.0), ys], axis=1)
    codes, scales = o.mx_quantize(blocks)
    assert np.all(scales == 127)
    np.testing.assert_array_equal(codes[:, 1:].ravel(), _e4m3_nearest_code(ys.ravel()))
    # (torch casts through fp32: compare values that fp32 holds exactly)
    low = (ys.ravel() < 448.0) & (ys.ravel().astype(np.float32) == ys.ravel())
    lib = torch.from_numpy(ys.ravel()[low].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes[:, 1:].ravel()[low], lib)
    # signs: the code of -v is the code of v with bit 7 set
    neg, _ = o.mx_quantize(-blocks)
    np.testing.assert_array_equal(neg, codes | 0x80)


def pin_mx_block_scale(o):
    """MX shared exponent s = floor(log2(max |v|)) - 8, clamped to [-127, 127], zero
    blocks s = -127 (E8M0 byte s + 127): closed forms; the block maximum's code lies in
    [256, 448]; each element is within half an E4M3 step (times 2^s) of its value; a
    block of E4M3 values times 2^s comes back exactly."""
    import oracle as orc
    rs = np.random.RandomState(43)
    for p in (-20, -8, -1, 0, 3, 9, 17):
        for f in (1.0, 1.37, 1.999):
            v = rs.uniform(-1, 1, 32) * (f * 2.0 ** p)
            v[rs.randint(32)] = -f * 2.0 ** p
            c, s = o.mx_quantize(v)
            assert int(s[0]) == p - 8 + 127, (p, f, s)
            q = orc.e4m3_value(c) * 2.0 ** (int(s[0]) - 127)
            assert 256.0 <= np.max(np.abs(orc.e4m3_value(c))) <= 448.0
            # each element within half the E4M3 spacing of its binade (2^(E-3), E >= -6),
            # times 2^s; a saturated element (|v| / 2^s in [448, 512)) is off by < 64 * 2^s
            a = np.abs(v) * 2.0 ** -(int(s[0]) - 127)
            E = np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -30))), -6)
            bound = np.where(a >= 448, 64.0, 2.0 ** (E - 4)) * 2.0 ** (int(s[0]) - 127)
            assert np.all(np.abs(q - v) <= bound * (1 + 1e-12)), (p, f)
    c, s = o.mx_quantize(np.zeros(32))
    assert s[0] == 0 and np.all(c == 0)
    c, s = o.mx_quantize(np.full(32, 2.0 ** -140))
    assert s[0] == 0
    c, s = o.mx_quantize(np.full(32, 2.0 ** 140))
    assert s[0] == 254
    exact = orc.e4m3_value(rs.randint(0, 127, 64).astype(np.uint8)) * 2.0 ** -5
    exact[0], exact[32] = 448 * 2.0 ** -5, -256 * 2.0 ** -5
    c, s = o.mx_quantize(exact)
    np.testing.assert_array_equal(orc.mxfp8_dequant(c[None], s[None])[0], exact)


def _mx_round_trip_np(v):
    """Quantise-dequantise along the last axis with the brute-force E4M3 rounding and
    the shared-exponent closed form (independent of the oracle's C code)."""
    import oracle as orc
    v = np.asarray(v, np.float64)
    b = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    amax = np.abs(b).max(axis=-1, keepdims=True)
    s = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, -127)
    s = np.clip(s, -127, 127)
    a = np.abs(b) * np.exp2(-s)
    q = orc.e4m3_value(_e4m3_nearest_code(a.ravel())).reshape(a.shape) * np.sign(b) * np.exp2(s)
    return q.reshape(v.shape)


def pin_mx_layer(o):
    """MXFP8 routed experts (mx_act): each routed expert computes on its MXFP8-rounded
    input row and MXFP8-rounded hidden row, shared experts on the plain row; checked
    against torch fp64 library ops fed by an independent quantiser, on tiny layers."""
    for act, bias in (("swiglu", False), ("gelu", True)):
        w = wl(n_tokens=6, d_model=64, d_ff=64, n_experts=4, top_k=2, act=act, has_bias=bias, n_shared=1,
               d_ff_shared=32, gating="softmax_topk")
        t = rand_layer(w, 47)
        cfg = o.config(w, mx_act=1)
        ow = o.weights(t)
        r = o.route(cfg, t["x"], ow)
        got = o.outputs(cfg, t["x"], ow, r)
        xq = torch.from_numpy(_mx_round_trip_np(t["x"].astype(np.float64)))
        ref = torch.from_numpy(torch_expert(t, 0, t["x"].astype(np.float64), act, bias, shared=True))
        for tok in range(w.n_tokens):
            for j in range(w.top_k):
                e = int(r["idx"][tok, j])
                W1 = torch.from_numpy(t["w1"][e].astype(np.float64))
                a = xq[tok] @ W1.T
                if act == "gelu":
                    hh = torch.nn.functional.gelu(a + torch.from_numpy(t["b1"][e].astype(np.float64)))
                else:
                    W3 = torch.from_numpy(t["w3"][e].astype(np.float64))
                    hh = torch.nn.functional.silu(a) * (xq[tok] @ W3.T)
                hq = torch.from_numpy(_mx_round_trip_np(hh.numpy()))
                y = hq @ torch.from_numpy(t["w2"][e].astype(np.float64)).T
                if act == "gelu":
                    y = y + torch.from_numpy(t["b2"][e].astype(np.float64))
                ref[tok] += float(r["gate"][tok, j]) * y
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-9, atol=1e-9)
        # and it differs from the unquantised layer (the rounding is really applied)
        plain = o.outputs(o.config(w), t["x"], ow, r)
        assert np.max(np.abs(plain - got)) > 1e-4


ALL_PINS = [pin_capacity, pin_router_logits, pin_softmax, pin_topk, pin_gates, pin_assign, pin_zero_router,
            pin_uniform_usage, pin_stats_formula, pin_single_expert_is_dense_ffn, pin_activation_zero,
            pin_brute_force, pin_dense_softmax_mixture, pin_expert_choice, pin_bf16_inputs_and_mimic,
            pin_page_entropy, pin_passthrough, pin_assign_shard, pin_mxfp8_dequant, pin_round_bf16_nearest_even,
            pin_e4m3_rounding, pin_mx_block_scale, pin_mx_layer]
