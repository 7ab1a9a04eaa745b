"""GPU-vs-oracle comparison for verification outputs.

Bar (written here, used by every parity test):
 - accepted lengths, emitted tokens and D-cut depths/offsets: bit-exact, except
 - an accept decision may differ only where |u - p/q| < 1e-6 (oracle's p/q);
   the request's comparison stops there (counted as an exemption);
 - the final token may differ only where u*S lies within 1e-6*S of the
   oracle's running sum C at the boundary between the two choices (counted);
 - p_j(x_j), q_j(x_j): relative error <= 1e-5 where the oracle value is
   >= 1e-30, absolute <= 1e-35 below that.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle as O

ACCEPT_BAND = 1e-6
FINAL_BAND = 1e-6
P_RTOL = 1e-5
P_TINY = 1e-30
P_ATOL_TINY = 1e-35


def to_host(batch):
    """numpy views of a VerifyBatch (bf16 as uint16 bit patterns)."""
    def arr(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return {
        "k": arr(batch.k), "cu": arr(batch.cu_draft), "target": arr(batch.target_logits),
        "draft": arr(batch.draft_logits), "tokens": arr(batch.draft_tokens),
        "u_accept": arr(batch.u_accept), "u_final": arr(batch.u_final),
    }


def subset(h, reqs, draft_stride=0):
    """Host arrays of the requests `reqs` only (packed or padded draft side kept)."""
    cu = h["cu"]
    k = h["k"]
    tr, dr, tok, ua = [], [], [], []
    for i in reqs:
        K = int(k[i])
        t0 = int(cu[i]) + i
        tr.append(h["target"][t0:t0 + K + 1])
        if draft_stride:
            d0 = i * draft_stride
            dr.append(h["draft"][d0:d0 + draft_stride])
            tok.append(h["tokens"][d0:d0 + draft_stride])
            ua.append(h["u_accept"][d0:d0 + draft_stride])
        else:
            d0 = int(cu[i])
            dr.append(h["draft"][d0:d0 + K])
            tok.append(h["tokens"][d0:d0 + K])
            ua.append(h["u_accept"][d0:d0 + K])
    ks = np.array([int(k[i]) for i in reqs], np.int32)
    V = h["target"].shape[1]
    return {
        "k": ks, "cu": np.concatenate([[0], np.cumsum(ks)]).astype(np.int32),
        "target": np.concatenate(tr) if tr else np.zeros((0, V), h["target"].dtype),
        "draft": np.concatenate(dr) if dr else np.zeros((0, V), h["target"].dtype),
        "tokens": np.concatenate(tok) if tok else np.zeros(0, np.int32),
        "u_accept": np.concatenate(ua) if ua else np.zeros(0, np.float32),
        "u_final": h["u_final"][list(reqs)],
    }


def oracle_run(h, temperature, draft_stride=0):
    if temperature == 0:
        return O.verify_greedy(h["target"], h["tokens"], h["cu"], draft_stride=draft_stride)
    return O.verify_sample(h["target"], h["draft"], h["tokens"], h["cu"], temperature,
                           h["u_accept"], h["u_final"], draft_stride=draft_stride)


def oracle_per_request(h, temperature, reqs, draft_stride=0, workers=None):
    """Oracle results for each request in `reqs`, one call per request on a
    thread pool (the C oracle releases the GIL)."""
    workers = workers or min(32, os.cpu_count() or 1)

    def one(i):
        return i, oracle_run(subset(h, [i], draft_stride), temperature, draft_stride)
    with ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(one, reqs))


def gpu_host(out, batch):
    return {k: out[k].detach().cpu().numpy() for k in ("tokens", "accept_len", "p", "q")}


class Report(dict):
    pass


def _draft_index(cu, i, j, stride):
    return i * stride + j if stride else int(cu[i]) + j


def compare_request(i, h, g, o, oi, temperature, draft_stride, rep):
    """Compare request i of the GPU outputs g (full-batch host arrays) with the
    oracle result o for that request (index oi inside o)."""
    K = int(h["k"][i])
    t0 = int(h["cu"][i]) + i
    ocu = o["_cu"]
    ot0 = int(ocu[oi]) + oi
    gl, ol = int(g["accept_len"][i]), int(o.accept_len[oi])
    gt = g["tokens"][t0:t0 + K + 1].tolist()
    ot = o.tokens[ot0:ot0 + K + 1].tolist()
    # probabilities (T > 0, every drafted position)
    if temperature > 0 and ol >= 0:
        for j in range(K):
            gd = _draft_index(h["cu"], i, j, draft_stride)
            od = _draft_index(ocu, oi, j, draft_stride)
            for name in ("p", "q"):
                ev = float(o[name][od])
                gv = float(g[name][gd])
                if ev >= P_TINY:
                    ok = abs(gv - ev) <= P_RTOL * ev
                else:
                    ok = abs(gv - ev) <= P_ATOL_TINY
                if not ok:
                    raise AssertionError(f"request {i} pos {j}: {name} gpu {gv!r} oracle {ev!r}")
                rep["max_rel_" + name] = max(rep.get("max_rel_" + name, 0.0),
                                             abs(gv - ev) / ev if ev >= P_TINY else 0.0)
    if gl == ol and gt == ot:
        return
    if temperature == 0 or ol < 0 or gl < 0:
        raise AssertionError(f"request {i}: gpu len {gl} tokens {gt}, oracle len {ol} tokens {ot}")
    if gl != ol:
        j = min(gl, ol)  # first position whose accept decision differs
        od = _draft_index(ocu, oi, j, draft_stride)
        u = float(h["u_accept"][_draft_index(h["cu"], i, j, draft_stride)])
        r = float(o.ratio[od])
        if abs(u - r) < ACCEPT_BAND and gt[:j] == ot[:j]:
            rep["exempt_accept"] = rep.get("exempt_accept", 0) + 1
            return
        raise AssertionError(f"request {i}: accept decision at {j} differs (u={u!r}, "
                             f"p/q={r!r}); gpu len {gl}, oracle len {ol}")
    # same accepted length, different final token: inverse-CDF boundary band
    a = gl
    if gt[:a] != ot[:a] or gt[a + 1:] != ot[a + 1:]:
        raise AssertionError(f"request {i}: accepted prefix differs: {gt} vs {ot}")
    y_g, y_o = gt[a], ot[a]
    uS, S = float(o.final[oi][0]), float(o.final[oi][1])
    st, C = O.final_cdf(o["_target"], o["_draft"], ocu, oi, a, temperature,
                        draft_stride=draft_stride)
    assert st == O.OK
    lo, hi = min(y_g, y_o), max(y_g, y_o)
    if y_g < 0:
        raise AssertionError(f"request {i}: gpu final token {y_g}")
    near = abs(C[hi - 1] - uS) <= FINAL_BAND * S and abs(C[lo] - uS) <= FINAL_BAND * S
    if near:
        rep["exempt_final"] = rep.get("exempt_final", 0) + 1
        return
    raise AssertionError(f"request {i}: final token gpu {y_g} oracle {y_o} (uS={uS}, "
                         f"C[lo]={C[lo]}, C[hi-1]={C[hi - 1]}, S={S})")


def compare_batch(batch, gpu_out, reqs=None, workers=None):
    """Compare GPU outputs against the oracle on requests `reqs` (all by
    default).  Returns a report with exemption counts."""
    h = to_host(batch)
    g = gpu_host(gpu_out, batch)
    B = batch.B
    reqs = list(range(B)) if reqs is None else list(reqs)
    stride = batch.draft_stride
    T = batch.temperature
    rep = Report(requests=len(reqs), exempt_accept=0, exempt_final=0)
    per = oracle_per_request(h, T, reqs, stride, workers)
    for i in reqs:
        o = per[i]
        sub = subset(h, [i], stride)
        o["_cu"] = sub["cu"]
        o["_target"] = sub["target"]
        o["_draft"] = sub["draft"]
        assert o.status == O.OK, (i, o.status)
        compare_request(i, h, g, o, 0, T, stride, rep)
    return rep
