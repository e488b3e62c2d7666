"""GPU-vs-oracle comparison helpers for the parity tests (test infrastructure).

``run_gpu`` runs one forward through the C ABI and copies every intermediate
out of the workspace; ``check`` feeds the oracle the same inputs (and, for the
routing, the GPU's own fp32 logits / probabilities) and compares:

* routing (top-k ids, ranks, drops, row numbering, expert offsets, counts): bit-exact
* gates, probabilities and statistics: relative 1e-5
* permuted rows: bit-exact copies of the token rows (MXFP8 layers: their codes and
  scales equal the oracle's quantisation of the token rows; H blocks obey the
  block rule)
* outputs: fp32 layers |y - y_ref| <= 1e-4 (|y_ref| + rms(y_ref)) per element;
  bf16 layers max |y - y_ref| <= 2e-2 rms(y_ref) (``raw_bar``, the workload
  shapes). The small coverage layers have heavy-tailed outputs (max |y_ref| up to
  15 rms) on which even the exact outputs rounded to bf16 miss that bar, so there
  it applies to the error beyond half a bf16 ulp of y_ref; the raw error is
  reported for every layer
* large layers: besides the sampled output tokens, the gate-scaled expert rows
  Yp (fp32, before the combine) of the first and last row of every expert
  segment and of the grouped GEMMs' ragged tiles (each last wave, the odd
  halves of CTA-pair tiles), and the shared experts' sum Ys, each against the
  oracle's expert applied to that row's token: max error <= 2e-2 of the row's rms
* the router logits themselves against the oracle's fp64-accumulated logits,
  and the oracle's self-routed choice, which may differ only at near-ties

The oracle is single-threaded code; the checker calls it for disjoint tokens
or rows from several host threads at once (each call runs in C with the
Python interpreter lock released) so the full-size checks stay short.
"""
from __future__ import annotations

import concurrent.futures
import os

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
    mx = getattr(w, "expert_weights", "bf16") == "mxfp8"
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
        # bf16 layers gather the up-projection's rows from x (no xp copy in the workspace);
        # MXFP8 layers hold the rows' E4M3 codes and E8M0 scales there (mx below)
        xp=v("xp", (R, d), dt).cpu()
        if not mx and lay.h - lay.xp >= R * d * (2 if dt == torch.bfloat16 else 4) else None,
        mx=tuple(a.cpu() for a in moe.mx_views(layer.cfg, layer.ws, "xp") + moe.mx_views(layer.cfg, layer.ws, "h"))
        if mx else None,
        stats=layer.read_stats(),
        capacity=C,
        # gate-scaled expert rows (fp32 [R, d]) and the shared experts' sum (fp32 [N, d])
        fetch_yp=lambda rows: v("yp", (R, d), torch.float32)[torch.as_tensor(rows, device=out.device)].cpu(),
        fetch_ys=(lambda toks: v("ys", (N, d), torch.float32)[torch.as_tensor(toks, device=out.device)].cpu())
        if w.n_shared > 0 else None,
    )
    return layer, t, res


def sample_tokens(N, n, seed=0):
    if n >= N:
        return np.arange(N, dtype=np.int64)
    rs = np.random.RandomState(seed)
    s = set(rs.choice(N, n - 2, replace=False).tolist()) | {0, N - 1}
    return np.array(sorted(s), dtype=np.int64)


def _oracle_array(t, n, experts=None):
    """Host copy of weight ``n`` as the oracle takes it (only ``experts`` of a routed
    stack if given). MXFP8 routed weights are given to the oracle as their exact
    dequantised values (bf16 bit patterns): the layer is defined on those."""
    from oracle import as_bf16_bits, mxfp8_dequant
    v = t[n]
    sel = None if experts is None else torch.as_tensor(experts, device=v.device, dtype=torch.long)
    if sel is not None and n in ("w1", "w3", "b1", "w2", "b2"):
        v = v[sel]
    if t.get(n + "_scale") is not None:
        sc = t[n + "_scale"] if sel is None else t[n + "_scale"][sel]
        return as_bf16_bits(mxfp8_dequant(v.cpu().numpy(), sc.cpu().numpy()))
    return torch_to_numpy(v)


def host_weights(t, experts=None):
    """numpy copies of the weights the oracle needs (only ``experts`` of the routed stack if given)."""
    h = {}
    for n, v in t.items():
        if v is None or n == "x" or n.endswith("_scale"):
            h[n] = None
            continue
        h[n] = _oracle_array(t, n, experts)
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


def n_threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def oracle_outputs_threaded(cfg, x_np, ow, routing, tokens):
    """o.outputs over disjoint chunks of ``tokens`` on several host threads."""
    o = oracle()
    tokens = np.asarray(tokens, np.int64)
    nt = n_threads()
    if tokens.size < 2 * nt:
        return o.outputs(cfg, x_np, ow, routing, tokens)
    parts = np.array_split(tokens, nt * 4)
    with concurrent.futures.ThreadPoolExecutor(nt) as ex:
        outs = list(ex.map(lambda p: o.outputs(cfg, x_np, ow, routing, p), parts))
    return np.concatenate(outs, axis=0)


def _host_arrays(t, names, experts=None):
    """numpy host copies of the named weight tensors (of the listed experts only, if given)."""
    h = {}
    for n in names:
        if t.get(n) is None:
            continue
        h[n] = _oracle_array(t, n, experts)
    return h


def _oracle_weights(h):
    """OracleWeights over host arrays; the caller keeps ``h`` alive while it is used."""
    from oracle import OracleWeights
    ow = OracleWeights()
    for name, _ in OracleWeights._fields_:
        a = h.get(name)
        assert a is None or a.flags["C_CONTIGUOUS"]
        setattr(ow, name, None if a is None else a.ctypes.data)
    return ow


def oracle_expert_terms(w, t, routed, shared_tokens):
    """The oracle's single-expert outputs E_e(x_t) (fp64 [d]) for the (expert, token)
    pairs in ``routed``, and sum_s shared_s(x_t) for ``shared_tokens``. Expert weights
    are copied to the host a chunk of experts at a time; the calls of a chunk run on
    several host threads."""
    o = oracle()
    routed = sorted(set((int(e), int(tok)) for e, tok in routed))
    shared_tokens = sorted(set(int(x) for x in shared_tokens))
    toks = sorted({tok for _, tok in routed} | set(shared_tokens))
    x = t["x"]
    xs = x[torch.as_tensor(toks, device=x.device, dtype=torch.long)].float().cpu().numpy().astype(np.float64)
    xrow = {tok: np.ascontiguousarray(xs[i]) for i, tok in enumerate(toks)}
    by_e = {}
    for e, tok in routed:
        by_e.setdefault(e, []).append(tok)
    experts = sorted(by_e)
    m = 3 if w.act == "swiglu" else 2
    per_expert = m * w.d_model * w.d_ff * (2 if w.dtype == "bf16" else 4)
    chunk = max(1, int(1.5e9 // per_expert))
    terms = {}
    with concurrent.futures.ThreadPoolExecutor(n_threads()) as ex:
        for c0 in range(0, len(experts), chunk):
            ce = experts[c0:c0 + chunk]
            h = _host_arrays(t, ("w1", "w3", "b1", "w2", "b2"), ce)
            cfg = o.config(w, n_experts=len(ce))
            ow = _oracle_weights(h)
            jobs = [(e, tok, i) for i, e in enumerate(ce) for tok in by_e[e]]
            ys = list(ex.map(lambda j: o.expert_apply(cfg, ow, j[2], xrow[j[1]]), jobs))
            for (e, tok, _), y in zip(jobs, ys):
                terms[(e, tok)] = y
            del h
        shared = {}
        if w.n_shared > 0 and shared_tokens:
            h = _host_arrays(t, ("ws1", "ws3", "bs1", "ws2", "bs2"))
            cfg = o.config(w)
            ow = _oracle_weights(h)

            def shared_sum(tok):
                acc = np.zeros(w.d_model)
                for s_ in range(w.n_shared):
                    acc += o.expert_apply(cfg, ow, s_, xrow[tok], shared=True)
                return acc

            for tok, y in zip(shared_tokens, ex.map(shared_sum, shared_tokens)):
                shared[tok] = y
            del h
    return terms, shared


def _pick_bn(swiglu, c0, c1):
    """The grouped GEMM's tile width: the largest of 256 / 128 / 64 whose output
    width (half of it for SwiGLU) divides the listed column counts."""
    for bn in (256, 128, 64):
        oc = bn // 2 if swiglu else bn
        if c0 % oc == 0 and (c1 <= 0 or c1 % oc == 0):
            return bn
    return 0


def ragged_tiles(w, expert_off, max_rows, sms):
    """Row ranges of the grouped GEMMs' ragged tiles, in the kernels' tile order
    (groups in order -- routed experts, then the shared experts --, inside a group
    column tile by column tile, row tiles innermost; tile i on CTA (pair) i mod W).
    Returns (routed ranges [(expert, lo, hi)] relative to the expert's segment,
    shared token ranges [(lo, hi)]): every tile of each launch's last, partly
    filled wave, and for CTA-pair tiles every 128-row half that ends a segment with
    an odd number of 128-row tiles."""
    BM = 128
    E, N, S = w.n_experts, w.n_tokens, w.n_shared
    m_e = np.diff(np.asarray(expert_off, np.int64))
    routed, shared = [], []

    def last_wave(groups, tile_rows, W):
        # groups: [(kind, id, m, n_tiles)]
        starts, total = [], 0
        for kind, gid, m, nt in groups:
            starts.append(total)
            total += -(-m // tile_rows) * nt
        if W <= 0 or total % W == 0:
            return
        first = (total // W) * W
        for (kind, gid, m, nt), s0 in zip(groups, starts):
            mtiles = -(-m // tile_rows)
            for tile in range(max(first, s0), s0 + mtiles * nt):
                mt = (tile - s0) % mtiles
                lo, hi = mt * tile_rows, min((mt + 1) * tile_rows, m)
                (routed.append((gid, lo, hi)) if kind == "e" else shared.append((lo, hi)))

    swiglu = w.act == "swiglu"
    # up-projection: single CTAs, 128-row tiles
    bn = _pick_bn(swiglu, w.d_ff, w.d_ff_shared if S > 0 else 0)
    oc = bn // 2 if swiglu else bn
    groups = [("e", e, int(m_e[e]), w.d_ff // oc) for e in range(E)] + \
             [("s", s_, N, w.d_ff_shared // oc) for s_ in range(S)]
    max_tiles = (max_rows // BM + E) * (w.d_ff // oc) + (S * -(-N // BM) * (w.d_ff_shared // oc) if S else 0)
    last_wave(groups, BM, min(max_tiles, sms))
    # down-projection: CTA pairs (256-row tiles) once experts average four 128-row tiles
    bn = _pick_bn(False, w.d_model, 0)
    pair = bn == 256 and max_rows >= 4 * BM * E
    nt = w.d_model // bn
    groups = [("e", e, int(m_e[e]), nt) for e in range(E)] + ([("s", 0, N, nt)] if S else [])
    if pair:
        max_pairs = (max_rows // (2 * BM) + E) * nt + (-(-N // (2 * BM)) * nt if S else 0)
        last_wave(groups, 2 * BM, min(max_pairs, sms // 2))
        for e in range(E):
            t128 = -(-int(m_e[e]) // BM)
            if t128 % 2 == 1:
                routed.append((e, (t128 - 1) * BM, int(m_e[e])))
        if S and (-(-N // BM)) % 2 == 1:
            shared.append(((-(-N // BM) - 1) * BM, N))
    else:
        max_tiles = (max_rows // BM + E) * nt + (-(-N // BM) * nt if S else 0)
        last_wave(groups, BM, min(max_tiles, sms))
    return routed, shared


def _pick_rows(lo, hi, rng, n_rand=2):
    rows = {lo, hi - 1}
    if hi - lo > 2:
        rows |= set(rng.randint(lo, hi, size=n_rand).tolist())
    return rows


def check_big_layer(w, t, res, r, tokens):
    """Full-size layers: the oracle's outputs of the sampled tokens, and row-level
    checks of the gate-scaled expert rows Yp and the shared sum Ys (see the module
    docstring). Returns (reference outputs of ``tokens``, report)."""
    N, E, k, d = w.n_tokens, w.n_experts, w.top_k, w.d_model
    ec = w.gating == "expert_choice"
    C = r["capacity"]
    rng = np.random.RandomState(1)
    # row -> (expert, token, oracle gate)
    if ec:
        sel, gec = r["sel"], r["gate_ec"]
        off = np.arange(E + 1, dtype=np.int64) * C

        def row_info(row):
            e, c = divmod(int(row), C)
            return e, int(sel[e, c]), float(gec[e, c])
    else:
        off = np.asarray(r["expert_off"], np.int64)
        row_of, idx, g = r["row_of"], r["idx"], r["gate"]
        inv = np.full(int(off[-1]), -1, np.int64)
        tt, jj = np.nonzero(row_of >= 0)
        inv[row_of[tt, jj]] = tt * k + jj

        def row_info(row):
            q = int(inv[int(row)])
            tok, j = divmod(q, k)
            return int(idx[tok, j]), tok, float(g[tok, j])
    # rows to check: segment ends + ragged tiles
    rows = set()
    for e in range(E):
        if off[e + 1] > off[e]:
            rows |= {int(off[e]), int(off[e + 1]) - 1}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rt, st = ragged_tiles(w, off, int(res["row_token"].size), sms)
    for e, lo, hi in rt:
        rows |= {int(off[e]) + x for x in _pick_rows(lo, hi, rng)}
    shared_tokens = set(tokens.tolist()) if w.n_shared > 0 else set()
    ys_tokens = set()
    if w.n_shared > 0:
        ys_tokens = {0, N - 1} | set(rng.randint(0, N, size=8).tolist())
        for lo, hi in st:
            ys_tokens |= _pick_rows(lo, hi, rng)
        shared_tokens |= ys_tokens
    rows = sorted(rows)
    infos = [row_info(x) for x in rows]
    # the sampled tokens' routed terms
    routed = set((e, tok) for e, tok, _ in infos)
    tok_terms = {}
    for tok in tokens.tolist():
        if ec:
            lst = [(e, float(gec[e, c])) for e in range(E) for c in np.flatnonzero(sel[e] == tok)]
        else:
            lst = [(int(idx[tok, j]), float(g[tok, j])) for j in range(k) if row_of[tok, j] >= 0]
        tok_terms[tok] = lst
        routed |= {(e, tok) for e, _ in lst}
    terms, shared = oracle_expert_terms(w, t, routed, shared_tokens)
    # outputs of the sampled tokens: shared sum first, then the routed terms in order
    ref = np.zeros((tokens.size, d))
    for i, tok in enumerate(tokens.tolist()):
        acc = shared[tok].copy() if w.n_shared > 0 else np.zeros(d)
        for e, gv in tok_terms[tok]:
            acc += gv * terms[(e, tok)]
        ref[i] = acc
    report = {}
    # gate-scaled expert rows, each against its own rms (the gates make rows differ in
    # size by orders of magnitude; their relative error comes from the bf16 hidden
    # activations and does not depend on the gate)
    yp_ref = np.stack([gv * terms[(e, tok)] for e, tok, gv in infos])
    yp_got = res["fetch_yp"](rows).numpy().astype(np.float64)
    row_rms = np.sqrt(np.mean(yp_ref ** 2, axis=1))
    ratio = np.max(np.abs(yp_got - yp_ref), axis=1) / np.maximum(row_rms, 1e-30)
    worst = int(np.argmax(ratio))
    assert ratio[worst] <= 2e-2, \
        f"expert row {rows[worst]} (expert {infos[worst][0]}): max err {ratio[worst]:.4f} of the row's rms"
    report["yp_rows_compared"] = len(rows)
    report["yp_max_err_over_row_rms"] = float(ratio[worst])
    if w.n_shared > 0:
        yt = sorted(ys_tokens)
        ys_ref = np.stack([shared[tok] for tok in yt])
        ys_got = res["fetch_ys"](yt).numpy().astype(np.float64)
        s_ratio = np.max(np.abs(ys_got - ys_ref), axis=1) / np.maximum(np.sqrt(np.mean(ys_ref ** 2, axis=1)), 1e-30)
        assert np.max(s_ratio) <= 2e-2, f"shared-expert row of token {yt[int(np.argmax(s_ratio))]} differs"
        report["ys_rows_compared"] = len(yt)
        report["ys_max_err_over_row_rms"] = float(np.max(s_ratio))
    return ref, report


def check_mx_rows(t, mx, row_token, rows_valid, max_rows_checked=4096):
    """MXFP8 layers: the permuted rows' codes and scales equal the oracle's MXFP8
    quantisation of their token rows (bit for bit: both quantise the same bf16
    values); the hidden rows H obey the block rule: each block's largest code lies in
    [256, 448] (a scale byte 0 block may hold less: its values are below 2^-119) and
    no code is NaN."""
    from oracle import e4m3_value
    o = oracle()
    xq, xs, hq, hs = mx
    n = min(rows_valid, max_rows_checked)
    rows = np.unique(np.concatenate([np.arange(min(n, rows_valid)),
                                     np.arange(max(0, rows_valid - 64), rows_valid)])).astype(np.int64)
    x = t["x"][torch.as_tensor(row_token[rows], device=t["x"].device, dtype=torch.long)]
    codes, scales = o.mx_quantize(x.float().cpu().numpy().astype(np.float64))
    got_c, got_s = xq[torch.as_tensor(rows)].numpy(), xs[torch.as_tensor(rows)].numpy()
    assert np.array_equal(got_s, scales), f"xp scale bytes differ in {np.count_nonzero(got_s != scales)} blocks"
    assert np.array_equal(got_c, codes), f"xp codes differ in {np.count_nonzero(got_c != codes)} elements"
    h = e4m3_value(hq[torch.as_tensor(rows)].numpy())
    assert not np.any(np.isnan(h)), "NaN code in H"
    hb = np.abs(h).reshape(len(rows), -1, 32).max(axis=2)
    sc = hs[torch.as_tensor(rows)].numpy()
    assert np.all(((hb >= 256) & (hb <= 448)) | (sc == 0)), "H block without a code in [256, 448]"
    return {"mx_rows_checked": int(len(rows))}


def check(w, t, res, n_sample=None, check_self_routed=True, raw_bar=False):
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
    # permuted rows are exact copies (layers that copy them; the gathering up-projection
    # reads x[row_token] itself, and row_token is compared above)
    if res["xp"] is not None:
        x = t["x"].detach().cpu()
        assert torch.equal(res["xp"][:rows_valid], x[torch.as_tensor(ref_row_token, dtype=torch.long)])
    if res.get("mx") is not None:
        report.update(check_mx_rows(t, res["mx"], ref_row_token, rows_valid))
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
        ref, rows_rep = check_big_layer(w, t, res, r, tokens)
        report.update(rows_rep)
    else:
        ow = o.weights(host_weights(t))
        ref = oracle_outputs_threaded(cfg, torch_to_numpy(t["x"]), ow, r, tokens)
    got = res["out"][torch.as_tensor(tokens)].float().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    if w.dtype == "f32":
        bound = 1e-4 * (np.abs(ref) + rms)
        assert np.all(err <= bound), f"fp32 output: worst excess {np.max(err - bound)}"
    else:
        # the error beyond half an ulp of the bf16 output (a bf16 output cannot be
        # nearer the exact value than that)
        excess = np.maximum(err - half_ulp_bf16(ref), 0.0)
        report["out_max_excess_over_rms"] = float(np.max(excess) / rms) if rms > 0 else 0.0
        if raw_bar:
            assert np.max(err) <= 2e-2 * rms, f"bf16 output: max err {np.max(err)} vs 2e-2*rms {2e-2 * rms}"
        else:
            assert np.max(excess) <= 2e-2 * rms, \
                f"bf16 output: max err beyond half an ulp {np.max(excess)} vs 2e-2*rms {2e-2 * rms}"
    report["out_max_err_over_rms"] = float(np.max(err) / rms) if rms > 0 else 0.0
    report["out_tokens_compared"] = int(tokens.size)
    if w.dtype == "bf16" and not big:
        # the same reference with bf16 stores where the pipeline has them (hidden
        # activations, output): what is left is fp32-vs-fp64 accumulation and
        # rounding flips
        cfg_m = o.config(w, mimic_bf16=1, capacity_factor=cfg.capacity_factor)
        ref_m = oracle_outputs_threaded(cfg_m, torch_to_numpy(t["x"]), ow, r, tokens)
        report["mimic_max_err_over_rms"] = float(np.max(np.abs(got - ref_m)) / rms) if rms > 0 else 0.0

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
