"""Device timeline of the decode-layer step, read from the instrumented library.

``python -m mxfp8_mlp_gqa_gb300.build --timeline`` builds ``libmxg_tl.so``: the same kernels,
compiled with ``-DMXG_TIMELINE``, whose decode-step kernels append one record per warp
{kernel id, block, warp, entry, return from the programmatic wait, exit, mark 1, mark 2}
(globaltimer ns) to a device buffer; the marks are kernel-specific phase points (GEMM: first
stage landed / accumulator complete, last MMA issued / split-K partials staged; attention:
first tile landed, last tile consumed; combine: merged, stores issued). ``bench.py --timeline`` replays the step's CUDA graph on that library and calls
:func:`summarize`, which folds the records of each step into launches (the step's kernel order
is fixed) and reports, per launch, when its first CTA entered, when the first warp came back
from the programmatic wait (its predecessor had completed), and when its last warp left.

The instrumented build adds a timer read and an atomic per warp, so its step is slightly
longer than the production library's; the timeline explains the bench's numbers, it does not
replace them.
"""
from __future__ import annotations

import ctypes

import numpy as np

KERNELS = {1: "mxfp8_quantize", 2: "rmsnorm_mxfp8_quantize", 3: "prev_tokens_shift", 4: "copy16",
           5: "kv_append", 6: "gqa_split", 7: "gqa_combine", 17: "mx_gemm_tc<split-K>",
           18: "mx_gemm_tc<SwiGLU>", 24: "mx_gemm_tc2"}
UNITS = ("attn", "gemm_tc", "quant", "small")

# the decode-layer step's launches in stream order: (kernel id, name of that launch); the
# prev-window shift runs on a forked graph branch and is listed first
STEP_ORDER = [(3, "prev_tokens_shift"), (2, "rmsnorm 1 + quant"), (17, "qkv gemm + kv append"),
              (6, "attention split"), (7, "attention combine"), (17, "o gemm + residual"),
              (2, "rmsnorm 2 + quant"), (18, "mlp gate/up + swiglu"), (17, "mlp down + residual")]


MAX_SM = 256  # regions of the device buffer, one per SM (kTlMaxSm)
REC = 6       # u64 per record (tl::kRec)


class Recorder:
    """Device buffer the instrumented kernels append to (attached to every unit of `lib`): one
    region of `cap` records and one counter per SM."""

    def __init__(self, lib, cap: int = 4096):
        import torch

        self.cap = cap
        self.buf = torch.zeros((MAX_SM, cap, REC), dtype=torch.int64, device="cuda")
        self.cnt = torch.zeros((MAX_SM,), dtype=torch.int32, device="cuda")
        for u in UNITS:
            f = getattr(lib, "mxg_tl_attach_" + u)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
            rc = f(ctypes.c_void_p(self.buf.data_ptr()), ctypes.c_void_p(self.cnt.data_ptr()), cap)
            if rc != 0:
                raise RuntimeError(f"mxg_tl_attach_{u} failed ({rc})")

    def reset(self):
        self.cnt.zero_()

    def records(self) -> np.ndarray:
        """[n, 8] int64: kernel id, block, warp, entry, wait return (0: none), exit, mark 1, mark 2."""
        cnt = np.minimum(self.cnt.cpu().numpy(), self.cap)
        buf = self.buf.cpu().numpy().view(np.uint64)
        r = np.concatenate([buf[sm, :c] for sm, c in enumerate(cnt)]) if cnt.sum() else np.zeros((0, REC), np.uint64)
        n = len(r)
        out = np.empty((n, 8), np.int64)
        out[:, 0] = (r[:, 0] >> np.uint64(48)).astype(np.int64)
        out[:, 1] = ((r[:, 0] >> np.uint64(16)) & np.uint64(0xFFFFFFFF)).astype(np.int64)
        out[:, 2] = (r[:, 0] & np.uint64(0xFFFF)).astype(np.int64)
        out[:, 3:] = r[:, 1:].astype(np.int64)
        return out


def split_launches(rec: np.ndarray, order=STEP_ORDER):
    """Assign one step's records to its launches: per kernel id, the records sorted by entry
    time are cut at the largest entry-time gaps into as many launches as the step has."""
    out = []
    for kid in sorted({k for k, _ in order}):
        names = [nm for k, nm in order if k == kid]
        r = rec[rec[:, 0] == kid]
        r = r[np.argsort(r[:, 3], kind="stable")]
        n = len(names)
        if len(r) == 0:
            continue
        if n > 1:
            gaps = np.diff(r[:, 3])
            cuts = np.sort(np.argsort(gaps)[-(n - 1):]) + 1
            parts = np.split(r, cuts)
        else:
            parts = [r]
        out += list(zip(names, parts))
    pos = {nm: i for i, (_, nm) in enumerate(order)}
    return sorted(out, key=lambda t: pos[t[0]])


def summarize(steps, order=STEP_ORDER):
    """Per launch: medians over the steps of CTAs, first entry, first wait return, median mark 1,
    last mark 2 and last exit (us from the step's first entry), and `exposed` = its last exit
    minus the last exit of the launch before it on the critical chain (the forked shift is off
    the chain)."""
    rows = {}
    for rec in steps:
        t0 = rec[:, 3].min()
        prev_end = None
        for name, r in split_launches(rec, order):
            w = r[:, 4][r[:, 4] > 0]
            ent = (r[:, 3].min() - t0) / 1e3
            wt = (w.min() - t0) / 1e3 if len(w) else float("nan")
            end = (r[:, 5].max() - t0) / 1e3
            m1 = r[:, 6][r[:, 6] > 0]
            m2 = r[:, 7][r[:, 7] > 0]
            d = rows.setdefault(name, {"ctas": [], "enter": [], "waited": [], "mark1": [], "mark2": [], "exit": [],
                                       "exposed": []})
            d["mark1"].append((np.median(m1) - t0) / 1e3 if len(m1) else float("nan"))
            d["mark2"].append((m2.max() - t0) / 1e3 if len(m2) else float("nan"))
            d["ctas"].append(len(np.unique(r[:, 1])))
            d["enter"].append(ent)
            d["waited"].append(wt)
            d["exit"].append(end)
            if name != "prev_tokens_shift":
                d["exposed"].append(end - (prev_end if prev_end is not None else 0.0))
                prev_end = end
    return {k: {kk: float(np.median(v)) if v else float("nan") for kk, v in d.items()} for k, d in rows.items()}


def format_table(summary, order=STEP_ORDER) -> str:
    lines = [f"{'launch':24s} {'CTAs':>6s} {'enter':>8s} {'waited':>8s} {'mark1':>8s} {'mark2':>8s} {'exit':>8s} "
             f"{'exposed':>8s}   (us)"]
    for _, name in order:
        if name not in summary:
            continue
        d = summary[name]
        lines.append(f"{name:24s} {d['ctas']:6.0f} {d['enter']:8.2f} {d['waited']:8.2f} {d['mark1']:8.2f} "
                     f"{d['mark2']:8.2f} {d['exit']:8.2f} {d['exposed']:8.2f}")
    return "\n".join(lines)
