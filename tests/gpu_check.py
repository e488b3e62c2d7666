"""GPU-vs-oracle comparison helpers for the parity tests (test infrastructure).

``run_gpu`` runs one forward through the C ABI and copies every intermediate
out of the workspace; ``check`` feeds the oracle the same inputs (and, for the
routing, the GPU's own fp32 logits / probabilities) and compares:

* routing (top-k ids, ranks, drops, row numbering, expert offsets, counts): bit-exact
* gates, probabilities and statistics: relative 1e-5
* permuted rows: bit-exact copies of the token rows
* outputs: fp32 layers |y - y_ref| <= 1e-4 (|y_ref| + rms(y_ref)) per element;
  bf16 layers max (|y - y_ref| - half a bf16 ulp of y_ref) <= 2e-2 rms(y_ref)
* the router logits themselves against the oracle's fp64-accumulated logits,
  and the oracle's self-routed choice, which may differ only at near-ties
"""
from __future__ import annotations

import numpy as np
import torch

import sparse_expert_ffn_softmax_b300 as moe
from oracle import Oracle, torch_to_numpy

_ORACLE = None


def oracle() -> Oracle:
    global _ORACLE
    if _ORACLE is None:
        _ORACLE = Oracle()
    return _ORACLE


def run_gpu(w, tensors=None, layer=None, repeat=1):
    t = tensors if tensors is not None else moe.make_inputs(w, "cuda")
    if layer is None:
        layer = moe.Layer(w, t)
    out = None
    for _ in range(repeat):
        out = layer.forward(t["x"])
    torch.cuda.synchronize()
    code, word = moe.get_device_status(layer.cfg, layer.ws)
    assert code == 0 and word == 0, (code, word)
    lay = layer.layout
    N, E, k, d = w.n_tokens, w.n_experts, w.top_k, w.d_model
    C = lay.capacity
    ec = w.gating == "expert_choice"
    sel_shape = (E, C) if ec else (N, k)
    R = lay.max_rows
    dt = w.torch_dtype
    v = layer.view
    res = dict(
        out=out.detach().cpu(),
        logits=v("logits", (N, E), torch.float32).cpu().numpy(),
        probs=v("probs", (N, E), torch.float32).cpu().numpy() if ec else None,
        idx=v("idx", sel_shape, torch.int32).cpu().numpy(),
        gate=v("gate", sel_shape, torch.float32).cpu().numpy(),
        tok_rows=v("tok_rows", (E * C,) if ec else (N, k), torch.int32).cpu().numpy(),
        tok_off=v("tok_off", (N + 1,), torch.int32).cpu().numpy() if ec else None,
        expert_off=v("expert_off", (E + 1,), torch.int32).cpu().numpy(),
        row_token=v("row_token", (R,), torch.int32).cpu().numpy(),
        row_gate=v("row_gate", (R,), torch.float32).cpu().numpy(),
        xp=v("xp", (R, d), dt).cpu(),
        stats=layer.read_stats(),
        capacity=C,
    )
    return layer, t, res


def sample_tokens(N, n, seed=0):
    if n >= N:
        return np.arange(N, dtype=np.int64)
    rs = np.random.RandomState(seed)
    s = set(rs.choice(N, n - 2, replace=False).tolist()) | {0, N - 1}
    return np.array(sorted(s), dtype=np.int64)


def host_weights(t, experts=None):
    """numpy copies of the weights the oracle needs (only ``experts`` of the routed stack if given)."""
    h = {}
    for n, v in t.items():
        if v is None or n == "x":
            h[n] = None
            continue
        if experts is not None and n in ("w1", "w3", "b1", "w2", "b2"):
            v = v[torch.as_tensor(experts, device=v.device, dtype=torch.long)]
        h[n] = torch_to_numpy(v)
    return h


def half_ulp_bf16(v):
    """Half the spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def rel_err(a, b, floor=1e-30):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.max(np.abs(a - b) / np.maximum(np.abs(b), floor)) if a.size else 0.0


def check(w, t, res, n_sample=None, check_self_routed=True):
    o = oracle()
    N, E, k, d = w.n_tokens, w.n_experts, w.top_k, w.d_model
    ec = w.gating == "expert_choice"
    # the library reads the capacity factor as an fp32; give the oracle the same value
    cfg = o.config(w, capacity_factor=float(np.float32(w.capacity_factor)))
    report = {}

    # ---- routing from the GPU's own logits: bit-exact -----------------------
    r = o.route(cfg, None, None, logits=res["logits"], ec_keys=res["probs"])
    C = r["capacity"]
    assert C == res["capacity"]
    st = res["stats"]
    if ec:
        assert np.array_equal(res["idx"], r["sel"]), "expert-choice selection differs"
        np.testing.assert_allclose(res["gate"], r["gate_ec"], rtol=1e-5, atol=1e-12)
        assert np.array_equal(res["expert_off"], np.arange(E + 1) * C)
        # token lists: each token's rows in ascending expert order
        tok_off, tok_rows = res["tok_off"], res["tok_rows"]
        cnt = np.zeros(N, np.int64)
        np.add.at(cnt, r["sel"].ravel(), 1)
        assert np.array_equal(np.diff(tok_off), cnt)
        rows_of_t = [[] for _ in range(N)]
        for e in range(E):
            for c_, tok in enumerate(r["sel"][e]):
                rows_of_t[tok].append(e * C + c_)
        ref_rows = np.array([x for tr in rows_of_t for x in tr], np.int32)
        assert np.array_equal(tok_rows, ref_rows)
        rows_valid = E * C
        ref_row_token = r["sel"].ravel()
    else:
        assert np.array_equal(res["idx"], r["idx"]), "top-k differs"
        assert np.array_equal(res["tok_rows"], r["row_of"]), "rows / drops differ"
        assert np.array_equal(res["expert_off"], r["expert_off"]), "expert offsets differ"
        assert np.array_equal(st["counts"].numpy(), r["counts"])
        assert np.array_equal(st["kept"].numpy(), r["kept"])
        assert st["dropped"] == r["dropped"]
        np.testing.assert_allclose(res["gate"], r["gate"], rtol=1e-5, atol=1e-12)
        rows_valid = int(r["expert_off"][-1])
        ref_row_token = np.empty(rows_valid, np.int64)
        ref_row_gate = np.empty(rows_valid, np.float64)
        for tt in range(N):
            for j in range(k):
                rr = r["row_of"][tt, j]
                if rr >= 0:
                    ref_row_token[rr] = tt
                    ref_row_gate[rr] = r["gate"][tt, j]
        np.testing.assert_allclose(res["row_gate"][:rows_valid], ref_row_gate, rtol=1e-5, atol=1e-12)
    assert st["rows"] == rows_valid and st["capacity"] == C
    assert np.array_equal(res["row_token"][:rows_valid], ref_row_token)
    # permuted rows are exact copies
    x = t["x"].detach().cpu()
    assert torch.equal(res["xp"][:rows_valid], x[torch.as_tensor(ref_row_token, dtype=torch.long)])
    # ---- statistics ---------------------------------------------------------
    ost = r["stats"]
    np.testing.assert_allclose(st["f"].numpy(), ost["f"], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(st["P"].numpy(), ost["P"], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(st["aux_loss"], ost["aux_loss"], rtol=1e-5)
    np.testing.assert_allclose(st["z_loss"], ost["z_loss"], rtol=1e-5)
    np.testing.assert_allclose(st["mean_lse_sq"], ost["mean_lse_sq"], rtol=1e-5)
    if ec:
        np.testing.assert_allclose(res["probs"], o.softmax(res["logits"])[0], rtol=1e-5, atol=1e-12)

    # ---- outputs on (sampled) tokens ----------------------------------------
    tokens = sample_tokens(N, n_sample or N)
    big = w.n_experts * w.d_ff * w.d_model > (1 << 27)
    if big:
        if ec:
            experts = sorted({e for e in range(E) if np.isin(r["sel"][e], tokens).any()})
        else:
            experts = sorted(set(r["idx"][tokens].ravel().tolist()))
        hw = host_weights(t, experts)
        remap = np.full(E, -1, np.int32)
        remap[experts] = np.arange(len(experts), dtype=np.int32)
        cfg_out = o.config(w, n_experts=len(experts), capacity_factor=cfg.capacity_factor)
        r_out = dict(r)
        if ec:
            r_out["sel"] = np.ascontiguousarray(r["sel"][experts])
            r_out["gate_ec"] = np.ascontiguousarray(r["gate_ec"][experts])
        else:
            r_out["idx"] = np.ascontiguousarray(remap[r["idx"]])
    else:
        hw = host_weights(t)
        cfg_out = cfg
        r_out = r
    ow = o.weights(hw)
    ref = o.outputs(cfg_out, torch_to_numpy(t["x"]), ow, r_out, tokens)
    got = res["out"][torch.as_tensor(tokens)].float().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    if w.dtype == "f32":
        bound = 1e-4 * (np.abs(ref) + rms)
        assert np.all(err <= bound), f"fp32 output: worst excess {np.max(err - bound)}"
    else:
        # A bf16 output cannot be nearer the exact value than half its own ulp; the
        # 2e-2 x rms bar applies to the error beyond that quantisation.
        half_ulp = half_ulp_bf16(ref)
        excess = np.maximum(err - half_ulp, 0.0)
        assert np.max(excess) <= 2e-2 * rms, \
            f"bf16 output: max err beyond half an ulp {np.max(excess)} vs 2e-2*rms {2e-2 * rms}"
    report["out_max_err_over_rms"] = float(np.max(err) / rms) if rms > 0 else 0.0
    if w.dtype == "bf16":
        # the same reference with bf16 stores where the pipeline has them (hidden
        # activations, output): what is left is fp32-vs-fp64 accumulation and
        # rounding flips
        cfg_m = o.config(w, mimic_bf16=1, n_experts=cfg_out.n_experts, capacity_factor=cfg.capacity_factor)
        ref_m = o.outputs(cfg_m, torch_to_numpy(t["x"]), ow, r_out, tokens)
        report["mimic_max_err_over_rms"] = float(np.max(np.abs(got - ref_m)) / rms) if rms > 0 else 0.0
        report["out_max_excess_over_rms"] = float(np.max(excess) / rms) if rms > 0 else 0.0

    # ---- router logits and the oracle's self-routed choice --------------------
    if check_self_routed:
        lt = tokens[: min(len(tokens), 64)]
        xs = torch_to_numpy(t["x"][torch.as_tensor(lt, device=t["x"].device)])
        wr = dict(w_router=torch_to_numpy(t["w_router"]),
                  logit_bias=None if t["logit_bias"] is None else torch_to_numpy(t["logit_bias"]))
        cfg_l = o.config(w, n_tokens=len(lt))
        L_own = o.router_logits(cfg_l, xs, o.weights(wr))
        L_gpu = res["logits"][lt]
        Lrms = float(np.sqrt(np.mean(L_own.astype(np.float64) ** 2)))
        assert np.max(np.abs(L_gpu - L_own)) <= 1e-4 * max(Lrms, 1e-30) + 1e-6 * np.max(np.abs(L_own))
        if not ec:
            idx_own = o.topk(L_own, k)
            for i in range(len(lt)):
                if set(idx_own[i]) != set(res["idx"][lt[i]]):
                    srt = np.sort(L_own[i])[::-1]
                    assert srt[k - 1] - srt[k] < 1e-4 * Lrms, f"token {lt[i]}: self-routed choice differs"
        report["logit_max_err"] = float(np.max(np.abs(L_gpu - L_own)))
    return report
