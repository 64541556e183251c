"""The all-reduce entry point that allocates nothing (coll_allreduce_static).

It is for callers that cannot allocate device memory when they need the collective: a
serving process that has already reserved its HBM for weights and the KV cache (a late
cudaMalloc would fail or fragment that reservation), or a loop that must not pay the
implicit device synchronisation of cudaMalloc/cudaFree. Its exchange buffers and flags live
in a fixed device array inside the library. These tests call it through the C ABI on two
calls in a row and compare every epoch's output with the CPU oracle (fixed rank-order
binary32 sum, one bf16 rounding: bit for bit), and with the plan-based path (coll_plan /
coll_run, dual-buffer protocol), which sums in the same order.

This file is named to be collected last.
"""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import collective_datapath_copy_gb300 as cdc  # noqa: E402
from collective_datapath_copy_gb300 import _lib  # noqa: E402
from collective_datapath_copy_gb300.build import build  # noqa: E402
from oracle import collectives  # noqa: E402
import synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    yield
    torch.cuda.synchronize()


def _arr(ts):
    return C.cast((C.c_void_p * len(ts))(*[t.data_ptr() for t in ts]), C.c_void_p)


def static_allreduce(ins, outs, count, dtype, n_epochs=1, in_stride=0, pool=1, out_stride=0,
                     status=None):
    return _lib.lib().coll_allreduce_static(
        len(ins), _lib.DTYPE[dtype], _arr(ins), _arr(outs), count, n_epochs, in_stride, pool,
        out_stride, C.c_void_p(status.data_ptr()) if status is not None else None,
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _host_inputs(seed, R, pool, n, dtype):
    """rows[r][p]: rank r's input of pool entry p (bf16 patterns or float32)."""
    rng = synth.seeded_rng(seed)
    gen = synth.normal_bf16 if dtype == "bf16" else synth.normal_f32
    return [np.stack([gen(rng, n) for _ in range(pool)]) for _ in range(R)]


def _to_dev(rows, dtype):
    tdt = torch.int16 if dtype == "bf16" else torch.float32
    return [torch.from_numpy(r.view(np.int16) if dtype == "bf16" else r).to("cuda").to(tdt)
            for r in rows]


def _inputs(seed, R, pool, n, dtype):
    return _to_dev(_host_inputs(seed, R, pool, n, dtype), dtype)


def _host(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == "bf16" else a


@pytest.mark.parametrize("R,n,dtype,epochs,pool", [(8, 4096, "bf16", 64, 7), (2, 1024, "f32", 3, 2),
                                                    (5, 1000, "bf16", 1, 1)])
def test_static_allreduce_matches_the_oracle_on_two_calls(R, n, dtype, epochs, pool):
    es = 2 if dtype == "bf16" else 4
    tdt = torch.int16 if dtype == "bf16" else torch.float32
    plan = cdc.Plan(cdc.allreduce(R, n, dtype), protocol="dual")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((31, 32)):
        rows = _host_inputs(seed, R, pool, n, dtype)
        ins = _to_dev(rows, dtype)
        ref = [torch.zeros(epochs, n, dtype=tdt, device="cuda") for _ in range(R)]
        got = [torch.full((epochs, n), 7, dtype=tdt, device="cuda") for _ in range(R)]
        code = static_allreduce(ins, got, n, dtype, epochs, n * es, pool, n * es, status)
        assert code == 0, f"call {call}: {code}"
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the oracle: epoch e of every rank is the rank-order sum of pool entry e % pool
        want = [collectives.allreduce([rows[r][e % pool] for r in range(R)], dtype)[0]
                for e in range(epochs)]
        for r in range(R):
            out = _host(got[r], dtype)
            for e in range(epochs):
                assert np.array_equal(out[e].view(np.uint8), want[e].view(np.uint8)), \
                    (call, r, e)
        # and the plan-based path, which sums in the same order
        plan.run(ins, ref, n_epochs=epochs, in_epoch_stride=n * es, in_pool=pool,
                 out_epoch_stride=n * es)
        assert plan.status()["code"] == 0
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"call {call}"
    plan.free()


def test_static_allreduce_rejects_what_does_not_fit():
    R, n = 8, 1 << 20  # 8 x 2 MiB: more than the fixed scratch array holds
    ins = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    outs = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    assert static_allreduce(ins, outs, n, "bf16") == _lib.D["COLL_ETOOBIG"]
    assert static_allreduce(ins, outs, 3, "bf16") == _lib.D["COLL_EALIGN"]
    # a count whose byte size wraps 64 bits is too big, not 16 bytes
    assert static_allreduce(ins, outs, (1 << 63) + 8, "bf16") == _lib.D["COLL_ETOOBIG"]


def test_python_binding_of_the_static_allreduce():
    # cdc.allreduce_static marshals the same call; errors surface as CollError
    R, n = 4, 2048
    rows = _host_inputs(41, R, 1, n, "bf16")
    ins = _to_dev(rows, "bf16")
    plan = cdc.Plan(cdc.allreduce(R, n, "bf16"), protocol="dual")
    ref = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, ref)
    assert plan.status()["code"] == 0
    got = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    assert cdc.allreduce_static(ins, got, n, "bf16") == 0
    torch.cuda.synchronize()
    want = collectives.allreduce([r[0] for r in rows], "bf16")[0]
    for a, b in zip(got, ref):
        assert np.array_equal(_host(a, "bf16"), want)
        assert torch.equal(a, b)
    big = [torch.zeros(1 << 20, dtype=torch.int16, device="cuda") for _ in range(8)]
    with pytest.raises(cdc.CollError):
        cdc.allreduce_static(big, [torch.zeros_like(b) for b in big], 1 << 20, "bf16")
    plan.free()
