"""ctypes view of libcoll.so (argument marshalling only; every step runs in the library).

The structures mirror include/coll.h field for field.
"""

from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libcoll.so")
HEADER = os.path.join(ROOT, "include", "coll.h")


def _header_defines():
    vals = {}
    with open(HEADER) as f:
        for line in f:
            m = re.match(r"#define\s+(COLL_\w+)\s+\(?(-?\d+)(?:ull)?\s*(?:<<\s*(\d+))?\)?", line)
            if m:
                v = int(m.group(2))
                if m.group(3):
                    v <<= int(m.group(3))
                vals[m.group(1)] = v
    return vals


D = _header_defines()
OK = D["COLL_OK"]
ERRNAMES = {v: k for k, v in D.items() if k.startswith("COLL_E")}

OP = {"copy": D["COLL_OP_COPY"], "sum": D["COLL_OP_SUM"]}
DTYPE = {"bf16": D["COLL_BF16"], "f32": D["COLL_F32"], "bytes": D["COLL_BYTES"]}
ESIZE = {"bf16": 2, "f32": 4, "bytes": 1}
PROTOCOL = {"barrier": D["COLL_PROTO_BARRIER"], "dual": D["COLL_PROTO_DUAL"],
            "spec": D["COLL_PROTO_SPEC"], "ll": D["COLL_PROTO_LL"]}
DATAPATH = {"oneshot": D["COLL_DP_ONESHOT"], "twoshot": D["COLL_DP_TWOSHOT"],
            "twoshot_pull": D["COLL_DP_TWOSHOT_PULL"]}
SPEC_CHECK = {"tagged": D["COLL_SPEC_TAGGED"], "literal": D["COLL_SPEC_LITERAL"],
              "relaxed": D["COLL_SPEC_TAGGED_RELAXED"]}
ORDER = {"rank": D["COLL_ORDER_RANK"], "tree": D["COLL_ORDER_TREE"]}
INJECT = {"skip_notify": D["COLL_INJECT_SKIP_NOTIFY"], "stagger": D["COLL_INJECT_STAGGER"],
          "spec_pause": D["COLL_INJECT_SPEC_PAUSE"]}

SEG_DTYPE = np.dtype([("rank", "<i4"), ("reserved", "<i4"), ("offset", "<u8"),
                      ("count", "<u8"), ("name", "<u8")])


class Config(C.Structure):
    _fields_ = [("protocol", C.c_int32), ("datapath", C.c_int32), ("zero_copy", C.c_int32),
                ("spec_check", C.c_int32), ("unit_bytes", C.c_int32),
                ("warps_per_rank", C.c_int32), ("ctas", C.c_int32), ("tile_bytes", C.c_int32),
                ("tma_min_bytes", C.c_uint64), ("spin_limit_ns", C.c_uint64),
                ("record_stamps", C.c_uint32), ("stamp_capacity", C.c_uint32),
                ("inject_flags", C.c_uint64), ("inject_seed", C.c_uint64),
                ("inject_rank", C.c_int32), ("inject_prob_ppm", C.c_uint32),
                ("inject_max_ns", C.c_uint64), ("inject_start_ns", C.c_uint64),
                ("inject_pause_ns", C.c_uint64), ("chain", C.c_int32),
                ("spec_delay_ns", C.c_int32), ("reduce_order", C.c_int32),
                ("reserved3", C.c_int32)]


class PlanInfo(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in ("n_names", "n_jobs", "n_tiles", "n_units", "n_warps",
                                          "min_bytes", "xbuf_bytes", "flag_bytes",
                                          "bulk_tile_bytes")]


class Stats(C.Structure):
    _fields_ = [("status", C.c_int32), ("fail_rank", C.c_int32), ("fail_unit", C.c_int32),
                ("fail_where", C.c_int32), ("fail_epoch", C.c_uint64), ("epochs", C.c_uint64),
                ("spec_checks", C.c_uint64), ("spec_retries", C.c_uint64)]


# entry point name -> (restype, argtypes)
_P = C.c_void_p
_SIGS = {
    "coll_config_default": (C.c_int, [C.POINTER(Config)]),
    "coll_plan": (C.c_int, [C.POINTER(_P), C.c_int, C.c_int, C.c_int, _P, C.c_size_t, _P, _P,
                            C.c_size_t, _P, C.POINTER(Config)]),
    "coll_validate": (C.c_int, [C.c_int, C.c_int, C.c_int, _P, C.c_size_t, _P, _P, C.c_size_t,
                                _P, C.POINTER(Config), C.POINTER(PlanInfo)]),
    "coll_plan_info": (C.c_int, [_P, C.POINTER(PlanInfo)]),
    "coll_run": (C.c_int, [_P, _P, _P, C.c_int, C.c_int64, C.c_int, C.c_int64, _P]),
    "coll_run_gemv": (C.c_int, [_P, _P, _P, C.c_int, _P, C.c_int, C.c_int64, C.c_int,
                                C.c_int64, _P]),
    "coll_status": (C.c_int, [_P, C.POINTER(Stats)]),
    "coll_stamps": (C.c_int64, [_P, _P, C.c_int64]),
    "coll_reset": (C.c_int, [_P]),
    "coll_free": (C.c_int, [_P]),
    "coll_strerror": (C.c_char_p, [C.c_int]),
    "coll_probe_flag_rtt": (C.c_int, [C.c_int, C.c_int, C.POINTER(C.c_uint64),
                                      C.POINTER(C.c_int), C.POINTER(C.c_int)]),
    "coll_allreduce_static": (C.c_int, [C.c_int, C.c_int, _P, _P, C.c_uint64, C.c_int,
                                        C.c_int64, C.c_int, C.c_int64, _P, _P]),
}

_lib = None


def lib():
    """Load libcoll.so (built by collective_datapath_copy_gb300.build). Raises if missing:
    there is no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with "
                              "`python -m collective_datapath_copy_gb300.build`")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


class CollError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = code
        msg = lib().coll_strerror(code).decode()
        super().__init__(f"{where}: {ERRNAMES.get(code, code)} ({msg})")


def check(code, where=""):
    if code != OK:
        raise CollError(code, where)
    return code


def make_config(**kw) -> Config:
    c = Config()
    lib().coll_config_default(C.byref(c))
    for k, v in kw.items():
        if v is None:
            continue
        if k == "protocol":
            v = PROTOCOL[v] if isinstance(v, str) else v
        elif k == "datapath":
            v = DATAPATH[v] if isinstance(v, str) else v
        elif k == "reduce_order":
            v = ORDER[v] if isinstance(v, str) else v
        elif k == "spec_check":
            v = SPEC_CHECK[v] if isinstance(v, str) else v
        elif k == "inject":
            k = "inject_flags"
            if isinstance(v, (list, tuple, set)):
                v = sum(INJECT[x] for x in v)
            elif isinstance(v, str):
                v = INJECT[v]
        elif k == "zero_copy":
            v = int(bool(v))
        if not hasattr(c, k):
            raise TypeError(f"unknown config field {k}")
        setattr(c, k, v)
    return c
