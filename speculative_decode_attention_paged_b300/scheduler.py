"""Binding of the host-side KV-aware AIMD rollout scheduler (include/s3r_sched.h).

Argument marshalling only: the scheduler runs in the library's C++ code.
"""

import ctypes

import numpy as np

from . import S3RError, load_library

AIMD, FIXED_OFFLOAD, RECOMPUTE = 0, 1, 2

_I32, _I64, _P = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p


class SchedConfig(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("pool_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("block_tokens", ctypes.c_int32), ("limit_init", ctypes.c_int32), ("limit_min", ctypes.c_int32),
                ("limit_max", ctypes.c_int32), ("add_step", ctypes.c_int32), ("mult", ctypes.c_double),
                ("util_low", ctypes.c_double), ("util_high", ctypes.c_double), ("backlog_max", ctypes.c_int32)]


class SchedTotals(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "tokens", "offloaded", "restored", "dropped", "recomputed",
                                               "preemptions", "peak_used", "running_sum")] + \
               [("stalled", ctypes.c_int32), ("limit_final", ctypes.c_int32)]


class SchedStep(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("ran", "admitted", "resumed", "limit", "paused", "pad")] + \
               [(n, ctypes.c_int64) for n in ("reserved", "used", "moved", "ctx_tokens")]


_STEP_KEYS = ("ran", "admitted", "resumed", "limit", "paused", "reserved", "used", "moved", "ctx_tokens")
_TOTAL_KEYS = ("steps", "tokens", "offloaded", "restored", "dropped", "recomputed", "preemptions", "peak_used",
               "running_sum", "stalled", "limit_final")

_SIG = {
    "s3r_sched_create": (ctypes.c_int, [ctypes.POINTER(SchedConfig), _I32, _P, _P, _P, _P, ctypes.POINTER(_P)]),
    "s3r_sched_step": (ctypes.c_int, [_P, ctypes.POINTER(SchedStep), _P, _I32, ctypes.POINTER(_I32),
                                      ctypes.POINTER(_I32)]),
    "s3r_sched_get_totals": (ctypes.c_int, [_P, ctypes.POINTER(SchedTotals)]),
    "s3r_sched_destroy": (None, [_P]),
    "s3r_sched_run": (ctypes.c_int, [ctypes.POINTER(SchedConfig), _I32, _P, _P, _P, _P, _I64,
                                     ctypes.POINTER(SchedStep), ctypes.POINTER(SchedTotals)]),
}


def _lib():
    lib = load_library()
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


def _check(name, status):
    if status != 0:
        raise S3RError(name, status)


def make_config(cfg):
    """SchedConfig from a dict with the fields of s3r_sched_config."""
    c = SchedConfig()
    for name, _ in SchedConfig._fields_:
        setattr(c, name, cfg.get(name, 0) if name not in ("mult", "util_low", "util_high") else float(cfg.get(name, 0.0)))
    return c


def _arrays(prompt_lens, response_lens, emits):
    p = np.ascontiguousarray(prompt_lens, dtype=np.int32)
    r = np.ascontiguousarray(response_lens, dtype=np.int32)
    lens = np.array([len(e) for e in emits], dtype=np.int64)
    off = np.zeros(len(emits) + 1, dtype=np.int64)
    np.cumsum(lens, out=off[1:])
    flat = np.ascontiguousarray(np.concatenate([np.asarray(e, dtype=np.int32) for e in emits])
                                if len(emits) else np.zeros(0, dtype=np.int32), dtype=np.int32)
    return p, r, off, flat


def _totals_dict(t):
    return {k: int(getattr(t, k)) for k in _TOTAL_KEYS}


def run(cfg, prompt_lens, response_lens, emits, max_steps=1_000_000, trace=True):
    """s3r_sched_run: (totals dict, list of step dicts or None)."""
    lib = _lib()
    p, r, off, flat = _arrays(prompt_lens, response_lens, emits)
    c = make_config(cfg)
    recs = (SchedStep * max_steps)() if trace else None
    tot = SchedTotals()
    _check("s3r_sched_run", lib.s3r_sched_run(ctypes.byref(c), len(p), p.ctypes.data, r.ctypes.data, off.ctypes.data,
                                              flat.ctypes.data, max_steps, recs, ctypes.byref(tot)))
    totals = _totals_dict(tot)
    steps = None
    if trace:
        steps = [{k: int(getattr(recs[i], k)) for k in _STEP_KEYS} for i in range(totals["steps"])]
    return totals, steps


class Scheduler:
    """Step-by-step handle: each step() returns its record and the ids of the
    requests in that round (the set an engine would run)."""

    def __init__(self, cfg, prompt_lens, response_lens, emits):
        self._lib = _lib()
        self._keep = _arrays(prompt_lens, response_lens, emits)
        p, r, off, flat = self._keep
        self.n = len(p)
        self._c = make_config(cfg)
        h = _P()
        _check("s3r_sched_create", self._lib.s3r_sched_create(ctypes.byref(self._c), self.n, p.ctypes.data,
                                                              r.ctypes.data, off.ctypes.data, flat.ctypes.data,
                                                              ctypes.byref(h)))
        self._h = h
        self._ids = np.zeros(max(self.n, 1), dtype=np.int32)
        self.finished = self.n == 0

    def step(self):
        rec, n_ran, fin = SchedStep(), _I32(0), _I32(0)
        _check("s3r_sched_step", self._lib.s3r_sched_step(self._h, ctypes.byref(rec), self._ids.ctypes.data,
                                                          len(self._ids), ctypes.byref(n_ran), ctypes.byref(fin)))
        self.finished = bool(fin.value)
        return {k: int(getattr(rec, k)) for k in _STEP_KEYS}, self._ids[:n_ran.value].copy()

    def totals(self):
        t = SchedTotals()
        _check("s3r_sched_get_totals", self._lib.s3r_sched_get_totals(self._h, ctypes.byref(t)))
        return _totals_dict(t)

    def close(self):
        if self._h:
            self._lib.s3r_sched_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
