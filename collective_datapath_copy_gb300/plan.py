"""Python face of the C ABI: compile a naming into a plan and run it on torch buffers.

PyTorch provides device memory and streams only; every step of a run (staging, flags,
copy, reduce) happens inside libcoll.so's kernels.
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from . import _lib
from ._lib import check, lib
from .namings import Naming


def _u64(vals) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(vals, dtype=np.uint64))


def _ptr(a: np.ndarray):
    return C.c_void_p(a.ctypes.data) if a.size else None


def validate(naming: Naming, **cfg) -> _lib.PlanInfo:
    """Host-side compile (no GPU needed). Raises CollError with the library's code."""
    info = _lib.PlanInfo()
    c = _lib.make_config(**cfg)
    il, ol = _u64(naming.in_len), _u64(naming.out_len)
    ins = np.ascontiguousarray(naming.in_segs)
    outs = np.ascontiguousarray(naming.out_segs)
    code = lib().coll_validate(naming.R, _lib.OP[naming.op], _lib.DTYPE[naming.dtype], _ptr(ins),
                               len(ins), _ptr(il), _ptr(outs), len(outs), _ptr(ol), C.byref(c),
                               C.byref(info))
    check(code, "coll_validate")
    return info


def validate_code(R, op, dtype, in_len, in_segs, out_len, out_segs, **cfg) -> int:
    """Return the library's validation code for raw arguments (for tests)."""
    c = _lib.make_config(**cfg)
    il, ol = _u64(in_len), _u64(out_len)
    ins = np.ascontiguousarray(in_segs)
    outs = np.ascontiguousarray(out_segs)
    return lib().coll_validate(R, op, dtype, _ptr(ins), len(ins), _ptr(il) if len(il) else None,
                               _ptr(outs), len(outs), _ptr(ol) if len(ol) else None,
                               C.byref(c), None)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(int(stream.cuda_stream))


def _dev_ptrs(tensors, R):
    arr = (C.c_void_p * R)()
    for r in range(R):
        t = tensors[r] if tensors is not None and r < len(tensors) else None
        arr[r] = None if t is None else t.data_ptr()
    return arr


def _check_buffers(R, tensors, used, nbytes, stride, count, where):
    """The library sees only addresses. Before a run, check that every buffer it will touch
    is a CUDA tensor whose storage holds all the bytes the run reads or writes there:
    nbytes[r] at each of `count` epochs spaced `stride` bytes apart. A tensor that is too
    small would otherwise be overrun on the device."""
    reach = int(stride) * (int(count) - 1) if count > 1 else 0
    for r in range(R):
        if not used[r]:
            continue
        t = tensors[r] if tensors is not None and r < len(tensors) else None
        if t is None:
            continue  # the library rejects a missing buffer itself
        if not t.is_cuda:
            raise ValueError(f"{where}: buffer of rank {r} is not a CUDA tensor")
        need = reach + int(nbytes[r])
        if reach >= 0 and need <= t.nbytes and t.is_contiguous():
            continue  # within the tensor's own bytes (the common case: no storage lookup)
        st = t.untyped_storage()
        s0, s1 = st.data_ptr(), st.data_ptr() + st.nbytes()
        lo = t.data_ptr() + min(0, reach)
        hi = t.data_ptr() + max(0, reach) + int(nbytes[r])
        if lo < s0 or hi > s1:
            raise _lib.CollError(_lib.D["COLL_EBOUNDS"],
                                 f"{where}: buffer of rank {r} holds {s1 - t.data_ptr()} bytes "
                                 f"from its start, the run touches [{lo - t.data_ptr()}, "
                                 f"{hi - t.data_ptr()})")


class Plan:
    """A compiled collective. Config keywords mirror coll_config_t (protocol='spec'|'dual'|
    'barrier', datapath='oneshot'|'twoshot', zero_copy, spec_check='tagged'|'literal', ...)."""

    def __init__(self, naming: Naming, **cfg):
        self.naming = naming
        self.cfg = dict(cfg)
        c = _lib.make_config(**cfg)
        il, ol = _u64(naming.in_len), _u64(naming.out_len)
        ins = np.ascontiguousarray(naming.in_segs)
        outs = np.ascontiguousarray(naming.out_segs)
        h = C.c_void_p()
        code = lib().coll_plan(C.byref(h), naming.R, _lib.OP[naming.op], _lib.DTYPE[naming.dtype],
                               _ptr(ins), len(ins), _ptr(il), _ptr(outs), len(outs), _ptr(ol),
                               C.byref(c))
        check(code, "coll_plan")
        self._h = h
        self._run_fn = lib().coll_run
        # what a run touches, per rank: the whole buffer of every rank that holds a segment
        # of a consumed name (inputs) or any output segment (outputs)
        es = _lib.ESIZE[naming.dtype]
        consumed = {int(x) for x in np.asarray(naming.out_segs["name"])}
        self._in_used = [False] * naming.R
        for row in naming.in_segs:
            if int(row["name"]) in consumed:
                self._in_used[int(row["rank"])] = True
        self._out_used = [False] * naming.R
        for row in naming.out_segs:
            self._out_used[int(row["rank"])] = True
        self._in_bytes = [int(x) * es for x in naming.in_len]
        self._out_bytes = [int(x) * es for x in naming.out_len]
        self.info = _lib.PlanInfo()
        check(lib().coll_plan_info(self._h, C.byref(self.info)), "coll_plan_info")

    def run(self, ins, outs, n_epochs=1, in_epoch_stride=0, in_pool=1, out_epoch_stride=0,
            stream=None):
        """Enqueue n_epochs epochs. ins/outs: per-rank torch CUDA tensors (or None for a
        rank without segments). Strides are in bytes."""
        R = self.naming.R
        self._check(ins, outs, n_epochs, in_epoch_stride, in_pool, out_epoch_stride)
        code = self._run_fn(self._h, C.cast(_dev_ptrs(ins, R), C.c_void_p),
                            C.cast(_dev_ptrs(outs, R), C.c_void_p), int(n_epochs),
                            int(in_epoch_stride), int(in_pool), int(out_epoch_stride),
                            _stream_handle(stream))
        if code:
            check(code, "coll_run")

    def _check(self, ins, outs, n_epochs, in_epoch_stride, in_pool, out_epoch_stride,
               in_bytes=None):
        R = self.naming.R
        _check_buffers(R, ins, self._in_used, in_bytes or self._in_bytes, in_epoch_stride,
                       in_pool, "coll_run")
        _check_buffers(R, outs, self._out_used, self._out_bytes, out_epoch_stride, n_epochs,
                       "coll_run")

    def bind(self, ins, outs, n_epochs=1, in_epoch_stride=0, in_pool=1, out_epoch_stride=0,
             stream=None):
        """Marshal a run once (buffers, strides, stream) and return a callable that enqueues
        it again: the per-call host cost is then the library call itself, which matters when
        small collectives are issued one by one on the same buffers."""
        return BoundRun(self, ins, outs, n_epochs, in_epoch_stride, in_pool, out_epoch_stride,
                        stream)

    def run_gemv(self, wts, xs, k, outs, n_epochs=1, x_epoch_stride=0, x_pool=1,
                 out_epoch_stride=0, stream=None):
        """Fused producer: each rank's payload is W_r x_r computed inside the engine.
        wts[r]: [k, in_len[r]] bf16 (W_r transposed); xs[r]: x vectors (k bf16 per epoch);
        k a multiple of 16, at most 8192 (coll_run_gemv has the full contract)."""
        R = self.naming.R
        self._check(xs, outs, n_epochs, x_epoch_stride, x_pool, out_epoch_stride,
                    in_bytes=[2 * int(k)] * R)
        _check_buffers(R, wts, self._in_used, [int(k) * b for b in self._in_bytes],
                       0, 1, "coll_run_gemv")
        code = lib().coll_run_gemv(self._h, C.cast(_dev_ptrs(wts, R), C.c_void_p),
                                   C.cast(_dev_ptrs(xs, R), C.c_void_p), int(k),
                                   C.cast(_dev_ptrs(outs, R), C.c_void_p), int(n_epochs),
                                   int(x_epoch_stride), int(x_pool), int(out_epoch_stride),
                                   _stream_handle(stream))
        check(code, "coll_run_gemv")

    def run_ptrs(self, in_ptrs, out_ptrs, n_epochs=1, in_epoch_stride=0, in_pool=1,
                 out_epoch_stride=0, stream=None):
        """Same as run() with raw device addresses (ints)."""
        R = self.naming.R
        ia = (C.c_void_p * R)(*[p or None for p in in_ptrs])
        oa = (C.c_void_p * R)(*[p or None for p in out_ptrs])
        return lib().coll_run(self._h, C.cast(ia, C.c_void_p), C.cast(oa, C.c_void_p),
                              int(n_epochs), int(in_epoch_stride), int(in_pool),
                              int(out_epoch_stride), _stream_handle(stream))

    def status(self) -> dict:
        st = _lib.Stats()
        code = lib().coll_status(self._h, C.byref(st))
        d = {f: getattr(st, f) for f, _ in _lib.Stats._fields_}
        d["code"] = code
        return d

    def stamps(self, n: int) -> np.ndarray:
        """Stamps of the last run: n+1 values (record_stamps=1) or 4n+1 (record_stamps=2)."""
        per = 4 if int(self.cfg.get("record_stamps", 0)) == 2 else 1
        buf = np.zeros(per * n + 1, dtype=np.uint64)
        m = lib().coll_stamps(self._h, C.c_void_p(buf.ctypes.data), per * n + 1)
        if m < 0:
            check(int(m), "coll_stamps")
        return buf[:m]

    def reset(self):
        check(lib().coll_reset(self._h), "coll_reset")

    def free(self):
        if getattr(self, "_h", None):
            lib().coll_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def probe_flag_rtt(peer_block: int = 1, iters: int = 20000):
    """Round trip (ns) of one flag ping-pong between two blocks, and their SM ids."""
    ns = C.c_uint64()
    a, b = C.c_int(), C.c_int()
    check(lib().coll_probe_flag_rtt(int(peer_block), int(iters), C.byref(ns), C.byref(a),
                                    C.byref(b)), "coll_probe_flag_rtt")
    return ns.value / iters, a.value, b.value


class BoundRun:
    """A run of a plan with its arguments marshalled once (see Plan.bind). Calling it
    enqueues the run again and raises CollError on a synchronous error. The buffers must stay
    alive and the stream valid while the object is used."""

    def __init__(self, plan, ins, outs, n_epochs, in_epoch_stride, in_pool, out_epoch_stride,
                 stream):
        R = plan.naming.R
        plan._check(ins, outs, n_epochs, in_epoch_stride, in_pool, out_epoch_stride)
        self._plan = plan
        self._keep = (list(ins), list(outs))  # keep the tensors alive
        self._ia = C.cast(_dev_ptrs(ins, R), C.c_void_p)
        self._oa = C.cast(_dev_ptrs(outs, R), C.c_void_p)
        self._args = (int(n_epochs), int(in_epoch_stride), int(in_pool), int(out_epoch_stride),
                      _stream_handle(stream))
        self._fn = lib().coll_run

    def __call__(self):
        code = self._fn(self._plan._h, self._ia, self._oa, *self._args)
        if code:
            check(code, "coll_run")


def allreduce_static(ins, outs, count, dtype="bf16", n_epochs=1, in_epoch_stride=0, in_pool=1,
                     out_epoch_stride=0, status=None, stream=None) -> int:
    """coll_allreduce_static: an all-reduce (fixed rank order, dual buffers) that allocates
    nothing, for callers that cannot allocate device memory at that point (HBM already
    reserved for weights and the KV cache; loops that must not pay cudaMalloc's implicit
    synchronisation); its exchange buffers and flags live in a fixed device array of the
    library, shared by every call, so calls must not overlap on the GPU. ins/outs:
    per-rank torch CUDA tensors of `count` elements; strides in bytes; `status`: optional
    int32 CUDA tensor that receives COLL_ETIMEDOUT if a bounded wait expires. Returns the
    library's code (raises on a synchronous error)."""
    R = len(ins)
    code = lib().coll_allreduce_static(
        R, _lib.DTYPE[dtype], C.cast(_dev_ptrs(ins, R), C.c_void_p),
        C.cast(_dev_ptrs(outs, R), C.c_void_p), int(count), int(n_epochs), int(in_epoch_stride),
        int(in_pool), int(out_epoch_stride),
        C.c_void_p(status.data_ptr()) if status is not None else None, _stream_handle(stream))
    check(code, "coll_allreduce_static")
    return code
