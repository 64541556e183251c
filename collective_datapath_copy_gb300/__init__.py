"""Collective datapath (copy / reduce) on one GB300, emulating R ranks on one GPU.

A collective is a naming of per-rank input and output segments plus copy or sum
(``namings``); ``Plan`` compiles it through the C ABI of libcoll.so (include/coll.h) and
runs it with the staged Stage/Notify/Consume engine (barrier, dual-buffer or speculative
protocol) or the zero-copy datapath. The library is required: there is no fallback.
"""

from . import namings  # noqa: F401
from ._lib import CollError, lib  # noqa: F401
from .namings import (Naming, allgather, allreduce, alltoall, alltoallv_from_routing,  # noqa: F401
                      broadcast, gather, moe_combine, moe_dispatch, reduce_scatter,
                      reduce_to_root, scatter, segs)
from .plan import Plan, allreduce_static, probe_flag_rtt, validate, validate_code  # noqa: F401
