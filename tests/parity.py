"""Shared GPU-vs-oracle comparison helpers (test infrastructure).

Tolerances
  * bias / logit / probe logit / matvec output: |gpu - oracle| <= 2e-3 + 1e-3 * |oracle|.
  * draft ids: bit-exact, except where the oracle's margin between its id and the GPU's
    id is within the fp32 rounding bound of the two logits (a near tie); the comparison
    then teacher-forces the oracle onto the GPU's id so one near tie does not fail every
    later position.  The bound for a logit base + sum_j w2[v,j] h[j] summed in fp32 in
    any order is (R + 2) * 2^-24 * (sum_j |w2[v,j] h[j]| + |base| + |bias|); the margin
    allowed is twice the sum of the two bounds.
  * probe gates: identical, except where |z_oracle - logit(t)| is within the value
    tolerance above (the GPU logit is checked to lie within it of the oracle's, so only
    inside that band can a correct fp32 evaluation land on the other side).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dspark_draft_sampling_gb300 import api

U32 = 2.0 ** -24
TOL_ABS, TOL_REL = 2e-3, 1e-3


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def within_tol(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > bound
    return (not bad.any()), float(err.max() if err.size else 0.0), int(bad.sum())


# ---------------------------------------------------------------- Markov draft ----------
def markov_to_device(inp, device="cuda"):
    d = dict(
        base=torch.from_numpy(np.ascontiguousarray(inp["base"])).to(device),
        w1=torch.from_numpy(inp["w1"].view(np.int16)).to(device),
        w2=torch.from_numpy(inp["w2"].view(np.int16)).to(device),
        d2t=None if inp["d2t"] is None else torch.from_numpy(inp["d2t"]).to(device),
        prev=torch.from_numpy(inp["prev0"].copy()).to(device),
    )
    return d


def gpu_markov(inp, *, dbg=True, dbg_bias=True, device="cuda", kernel="auto"):
    t = markov_to_device(inp, device)
    B, k, V = t["base"].shape
    R = t["w2"].shape[1]
    dl = torch.full_like(t["base"], float("nan")) if dbg else None
    db = torch.full_like(t["base"], float("nan")) if (dbg and dbg_bias) else None
    ws = api.new_markov_workspace(B, k, V, R, device)
    out = api.markov_draft(t["base"], t["w1"], t["w2"], t["d2t"], t["prev"], dbg_logits=dl,
                           dbg_bias=db, workspace=ws, kernel=kernel)
    status = api.markov_status(ws)
    return dict(out_ids=out.cpu().numpy(), prev=t["prev"].cpu().numpy(),
                logits=None if dl is None else dl.cpu().numpy(),
                bias=None if db is None else db.cpu().numpy(), status=status)


def draft_from_target(inp, out_ids):
    if inp["d2t"] is None:
        return out_ids.copy()
    d2t = inp["d2t"].astype(np.int64)
    inv = np.full(int(d2t.max()) + 1, -1, np.int64)
    inv[d2t] = np.arange(len(d2t))
    return inv[out_ids]


def near_tie_bound(inp, r, i, prev, v):
    R = inp["w2"].shape[1]
    h = bf16_to_f64(inp["w1"][prev])
    prod = bf16_to_f64(inp["w2"][v]) * h
    a = np.abs(prod).sum() + abs(float(inp["base"][r, i, v])) + abs(prod.sum())
    return (R + 2) * U32 * a


def check_markov(inp, g, *, values=True):
    """Assert GPU Markov results match the oracle; returns a small report dict."""
    assert g["status"] == 0, f"device status {g['status']}"
    gd = draft_from_target(inp, g["out_ids"])
    B, k, V = inp["base"].shape
    assert np.all((gd >= 0) & (gd < V)), "GPU id outside the draft vocabulary"
    want_bias = values and g.get("bias") is not None
    o = oracle.markov_draft(inp["base"], inp["w1"], inp["w2"], inp["d2t"], inp["prev0"],
                            forced_prev=gd, want_logits=True, want_bias=want_bias)
    L = o["logits"]
    exempt = []
    for r, i in np.argwhere(o["draft_ids"] != gd):
        ov, gv = int(o["draft_ids"][r, i]), int(gd[r, i])
        p = int(inp["prev0"][r]) if i == 0 else int(gd[r, i - 1])
        margin = L[r, i, ov] - L[r, i, gv]
        bound = 2 * (near_tie_bound(inp, r, i, p, ov) + near_tie_bound(inp, r, i, p, gv))
        assert margin <= bound, (f"request {r} position {i}: GPU id {gv} vs oracle {ov}, "
                                 f"margin {margin:.3e} > rounding bound {bound:.3e}")
        exempt.append((int(r), int(i), ov, gv, float(margin)))
    exempt_set = {(e[0], e[1]) for e in exempt}
    for r in range(B):
        for i in range(k):
            if (r, i) not in exempt_set:
                assert g["out_ids"][r, i] == o["out_ids"][r, i]
    np.testing.assert_array_equal(g["prev"], gd[:, -1])
    rep = dict(n_exempt=len(exempt), exempt=exempt)
    if values and g.get("logits") is not None:
        ok, err, nbad = within_tol(g["logits"], L)
        assert ok, f"{nbad} logits outside tolerance (max err {err:.3e})"
        rep["max_logit_err"] = err
    if want_bias:
        ok, err, nbad = within_tol(g["bias"], o["bias"])
        assert ok, f"{nbad} bias values outside tolerance (max err {err:.3e})"
        rep["max_bias_err"] = err
    return rep


# ---------------------------------------------------------------- confidence probe ------
def gpu_probe(inp, device="cuda"):
    wq = torch.from_numpy(inp["wq"]).to(device)
    hid = torch.from_numpy(np.ascontiguousarray(inp["hidden"])).to(device)
    z, gate = api.conf_probe(wq, hid, inp["bias"], inp["threshold"])
    return z.cpu().numpy(), gate.cpu().numpy()


def check_probe(inp, z, gate):
    zo, go = oracle.conf_probe(inp["wq"], inp["hidden"], inp["bias"], inp["threshold"])
    ok, err, nbad = within_tol(z, zo)
    assert ok, f"{nbad} probe logits outside tolerance (max err {err:.3e})"
    t = inp["threshold"]
    thr = np.log(t / (1 - t))
    near = np.abs(zo - thr) <= TOL_ABS + TOL_REL * abs(thr)
    mism = (gate != go) & ~near
    assert not mism.any(), f"{int(mism.sum())} gate decisions differ"
    return dict(max_z_err=err, n_near_threshold=int(near.sum()),
                n_gate_mismatch=int((gate != go).sum()))


# ---------------------------------------------------------------- WS matvec -------------
def check_ws(inp, y32=None, y16=None, exact=False):
    """WS matvec outputs against the fp64 oracle: within the value tolerance; the fp16 output
    is the RNE of the fp32 one.  With exact=True (inputs whose every partial sum is exact in
    fp32, so any correct fp32 accumulation gives Y itself) the fp32 output must equal Y and
    the fp16 output the oracle's RNE(Y), bit for bit."""
    Y, Y16 = oracle.ws_matvec(inp["W"], inp["X"])
    rep = {}
    if y32 is not None:
        ok, err, nbad = within_tol(y32, Y)
        assert ok, f"{nbad} fp32 outputs outside tolerance (max err {err:.3e})"
        if exact:
            np.testing.assert_array_equal(np.asarray(y32, np.float64), Y)
        rep["max_err_fp32"] = err
    if y16 is not None:
        yf = y16.view(np.float16).astype(np.float64)
        ok, err, nbad = within_tol(yf, Y)
        assert ok, f"{nbad} fp16 outputs outside tolerance (max err {err:.3e})"
        if y32 is not None:
            # both outputs come from the same fp32 sum: the fp16 one must be its RNE
            np.testing.assert_array_equal(y16, y32.astype(np.float32).astype(np.float16)
                                          .view(np.uint16))
        if exact:
            np.testing.assert_array_equal(y16, Y16)
        rep["fp16_exact_rne"] = int((y16 == Y16).sum())
        rep["fp16_total"] = int(y16.size)
    return rep


def check_ws_q8(inp, y32=None, y16=None):
    """Quantized matvec outputs against the fp64 oracle (same tolerance as the fp16 matvec)."""
    Y = oracle.ws_matvec_q8(inp["Wq8"], inp["X"])
    rep = {}
    if y32 is not None:
        ok, err, nbad = within_tol(y32, Y)
        assert ok, f"{nbad} fp32 outputs outside tolerance (max err {err:.3e})"
        rep["max_err_fp32"] = err
    if y16 is not None:
        yf = y16.view(np.float16).astype(np.float64)
        ok, err, nbad = within_tol(yf, Y)
        assert ok, f"{nbad} fp16 outputs outside tolerance (max err {err:.3e})"
        if y32 is not None:
            np.testing.assert_array_equal(y16, y32.astype(np.float32).astype(np.float16)
                                          .view(np.uint16))
    return rep
