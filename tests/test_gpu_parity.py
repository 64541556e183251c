"""GPU parity: every datapath and protocol of libcoll.so against the CPU oracle.

Copies and fixed-order sums must be bit-exact. Inputs are the seeded synthetic workloads
(uniform[-1,1] / N(0,1) bf16 or fp32 values, Zipf routing tables) at sizes the oracle
finishes in seconds, plus full-size cases checked in full or on samples.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import collective_datapath_copy_gb300 as cdc  # noqa: E402
from collective_datapath_copy_gb300 import namings  # noqa: E402
from collective_datapath_copy_gb300.build import build  # noqa: E402
from oracle import collectives, naming as onaming  # noqa: E402
from oracle.arith import NPTYPE  # noqa: E402
import synth  # noqa: E402

from gpu_util import bits_equal, empty_dev, from_dev, to_dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()


def gen(dist, rng, n, dtype):
    if dtype == "bytes":
        return synth.random_bytes(rng, n)
    if dtype == "f32":
        return synth.uniform_f32(rng, n) if dist == "uniform" else synth.normal_f32(rng, n)
    return synth.uniform_bf16(rng, n) if dist == "uniform" else synth.normal_bf16(rng, n)


def oracle_outputs(nm, ins, init=None):
    outs = [np.zeros(n, dtype=NPTYPE[nm.dtype]) if init is None else init[r].copy()
            for r, n in enumerate(nm.out_len)]
    assert onaming.run_naming(nm.R, nm.op, nm.dtype, nm.in_len, nm.rows("in"), nm.out_len,
                              nm.rows("out"), ins, outs) == 0
    return outs


def run_once(nm, ins_np, **cfg):
    """One epoch through the C ABI; returns (per-rank outputs, canary-initialised copy)."""
    plan = cdc.Plan(nm, **cfg)
    ins = [to_dev(x, nm.dtype) for x in ins_np]
    outs = [empty_dev(n, nm.dtype) for n in nm.out_len]
    init = [from_dev(o, nm.dtype).copy() for o in outs]
    plan.run(ins, outs)
    st = plan.status()
    assert st["code"] == 0, st
    res = [from_dev(o, nm.dtype) for o in outs]
    plan.free()
    return res, init


DATAPATHS = [
    dict(zero_copy=1, datapath="oneshot"),
    dict(zero_copy=1, datapath="twoshot"),
    dict(protocol="barrier"),
    dict(protocol="dual"),
    dict(protocol="spec"),
    dict(protocol="spec", datapath="twoshot"),
    dict(protocol="barrier", datapath="twoshot"),
    dict(protocol="spec", datapath="twoshot_pull"),
    dict(protocol="barrier", datapath="twoshot_pull"),
]


# ------------------------------------------------------------ small all-reduce (R=2, f32)

@pytest.mark.parametrize("cfg", DATAPATHS, ids=lambda c: "-".join(f"{k}={v}" for k, v in c.items()))
def test_allreduce_r2_f32_1024(cfg):
    rng = synth.seeded_rng(1)
    xs = [synth.uniform_f32(rng, 1024) for _ in range(2)]
    nm = namings.allreduce(2, 1024, "f32")
    got, _ = run_once(nm, xs, **cfg)
    want = collectives.allreduce(xs, "f32")
    for g, w in zip(got, want):
        assert bits_equal(g, w)


# ------------------------------------------------------------ collectives, several sizes

SIZES_B = [1024, 4096, 65536, 1 << 20]


@pytest.mark.parametrize("msg_bytes", SIZES_B)
@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter", "allgather", "broadcast", "alltoall"])
@pytest.mark.parametrize("mode", ["zc-oneshot", "zc-twoshot", "staged-spec"])
def test_collective_sweep_r8_bf16(kind, msg_bytes, mode):
    R = 8
    n = msg_bytes // 2
    rng = synth.seeded_rng(3)
    xs = [synth.uniform_bf16(rng, n) for _ in range(R)]
    nm = getattr(namings, kind)(R, n, "bf16")
    cfg = {"zc-oneshot": dict(zero_copy=1, datapath="oneshot"),
           "zc-twoshot": dict(zero_copy=1, datapath="twoshot"),
           "staged-spec": dict(protocol="spec")}[mode]
    got, _ = run_once(nm, xs, **cfg)
    if kind == "allreduce":
        want = collectives.allreduce(xs, "bf16")
    elif kind == "reduce_scatter":
        want = collectives.reduce_scatter(xs, "bf16")
    elif kind == "allgather":
        want = collectives.allgather(xs)
    elif kind == "broadcast":
        want = collectives.broadcast(xs, 0)
    else:
        want = collectives.alltoall(xs)
    for g, w in zip(got, want):
        assert bits_equal(g, w)


# ------------------------------------------------------------ random namings, edge cases

@pytest.mark.parametrize("seed", range(24))
def test_random_namings_zero_copy(seed):
    op = "copy" if seed % 3 == 0 else "sum"
    dtype = ["bf16", "f32", "bytes"][seed % 3] if op == "copy" else ["bf16", "f32"][seed % 2]
    R = 1 + seed % 5
    rng = synth.seeded_rng(900 + seed)
    il, i, ol, o = synth.random_naming(rng, R, 3000, 5, 4, op)
    nm = namings.Naming(R, op, dtype, il, namings.segs(i), ol, namings.segs(o))
    xs = [gen("normal", rng, n, dtype) for n in il]
    got, init = run_once(nm, xs, zero_copy=1, datapath="twoshot" if seed % 2 else "oneshot")
    want = oracle_outputs(nm, xs, init)  # unnamed elements keep the canary
    for g, w in zip(got, want):
        assert bits_equal(g, w)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("protocol", ["barrier", "dual", "spec", "ll"])
def test_random_namings_staged(seed, protocol):
    # staged plans need 16-byte-aligned segments: scale a random naming by 8 elements
    op = "copy" if seed % 3 == 0 else "sum"
    dtype = "bf16"
    R = 1 + seed % 6
    rng = synth.seeded_rng(1200 + seed)
    il, i, ol, o = synth.random_naming(rng, R, 200, 4, 4, op)
    k = 8
    il = [x * k for x in il]
    ol = [x * k for x in ol]
    i = [(r, off * k, c * k, nmv) for (r, off, c, nmv) in i]
    o = [(r, off * k, c * k, nmv) for (r, off, c, nmv) in o]
    nm = namings.Naming(R, op, dtype, il, namings.segs(i), ol, namings.segs(o))
    xs = [gen("normal", rng, n, dtype) for n in il]
    dp = ["oneshot", "twoshot", "twoshot_pull"][seed % 3]
    if protocol == "ll" and dp == "twoshot_pull":
        dp = "twoshot"
    got, init = run_once(nm, xs, protocol=protocol, datapath=dp)
    want = oracle_outputs(nm, xs, init)
    for g, w in zip(got, want):
        assert bits_equal(g, w)


def test_many_producers_and_ragged_tail():
    # 17 producers (more than one batch of 8 loads), n not a multiple of any tile
    R, n = 17, 12345
    rng = synth.seeded_rng(77)
    xs = [synth.normal_f32(rng, n) * np.float32(2.0) ** rng.integers(-10, 10, n).astype(np.float32)
          for _ in range(R)]
    nm = namings.allreduce(R, n, "f32")
    for cfg in (dict(zero_copy=1), dict(zero_copy=1, datapath="twoshot", tile_bytes=4096)):
        got, _ = run_once(nm, xs, **cfg)
        want = collectives.allreduce(xs, "f32")
        for g, w in zip(got, want):
            assert bits_equal(g, w)


def test_misaligned_zero_copy_segments_use_the_elementwise_path():
    R, n = 3, 1001
    rng = synth.seeded_rng(78)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    i = [(r, 1 + r, 997, 5) for r in range(R)]
    o = [(r, 3, 997, 5) for r in range(R)]
    nm = namings.Naming(R, "sum", "bf16", [n] * R, namings.segs(i), [n] * R, namings.segs(o))
    got, init = run_once(nm, xs, zero_copy=1)
    want = oracle_outputs(nm, xs, init)
    for g, w in zip(got, want):
        assert bits_equal(g, w)


def test_empty_naming_and_single_rank():
    nm = namings.Naming(2, "sum", "bf16", [16, 16], namings.segs([]), [16, 16], namings.segs([]))
    for cfg in (dict(zero_copy=1), dict(protocol="spec")):
        got, init = run_once(nm, [np.zeros(16, np.uint16)] * 2, **cfg)
        for g, w in zip(got, init):
            assert bits_equal(g, w)
    rng = synth.seeded_rng(79)
    x = synth.random_bytes(rng, 4096)
    got, _ = run_once(namings.broadcast(1, 4096, "bytes"), [x], zero_copy=1)
    assert bits_equal(got[0], x)


def test_special_values_sum():
    # signed zeros, subnormals, overflow to inf; NaN compared as a class (payloads of NaN
    # are not fixed by IEEE 754 and differ between host and device adders)
    vals = np.array([0x8000, 0x8000, 0x0001, 0x7F7F, 0x3F80, 0xBF80, 0x0000, 0x7FC0], np.uint16)
    R = 2
    a = np.tile(vals, 64)
    b = np.tile(np.array([0x8000, 0x0000, 0x0001, 0x7F7F, 0xBF80, 0x3F80, 0x8000, 0x3F80],
                         np.uint16), 64)
    nm = namings.allreduce(R, a.size, "bf16")
    for cfg in (dict(zero_copy=1), dict(protocol="spec")):
        got, _ = run_once(nm, [a, b], **cfg)
        want = collectives.allreduce([a, b], "bf16")
        g = got[0]
        w = want[0]
        nan_g = (g & 0x7FFF) > 0x7F80
        nan_w = (w & 0x7FFF) > 0x7F80
        assert np.array_equal(nan_g, nan_w)
        assert np.array_equal(g[~nan_g], w[~nan_w])


# ------------------------------------------------------------ decode all-reduce epochs

def _decode_case(R=8, n=4096, pool=7, seed=2):
    rng = synth.seeded_rng(seed)
    pool_np = [[synth.normal_bf16(rng, n) for _ in range(R)] for _ in range(pool)]
    ins = [torch.stack([to_dev(pool_np[p][r], "bf16") for p in range(pool)]).contiguous()
           for r in range(R)]
    expect = [collectives.allreduce(pool_np[p], "bf16")[0] for p in range(pool)]
    expect_dev = torch.stack([to_dev(e, "bf16") for e in expect])  # [pool, n]
    return ins, expect_dev


def _check_epochs(outs, expect_dev, n_epochs, pool):
    """outs[r]: [n_epochs, n] device tensors; epoch i must equal expect[i % pool]."""
    idx = torch.arange(n_epochs, device="cuda") % pool
    want = expect_dev[idx]
    bad = 0
    for o in outs:
        bad += int((o != want).any(dim=1).sum())
    return bad


@pytest.mark.parametrize("cfg", [
    dict(protocol="spec"),
    dict(protocol="spec", spec_check="tagged"),
    dict(protocol="spec", spec_check="tagged", inject="stagger", inject_seed=11,
         inject_prob_ppm=100000, inject_max_ns=20000, inject_start_ns=5000),
    dict(protocol="spec", spec_check="relaxed", inject="stagger", inject_seed=12,
         inject_prob_ppm=100000, inject_max_ns=20000, inject_start_ns=5000),
    dict(protocol="ll", inject="stagger", inject_seed=13, inject_prob_ppm=100000,
         inject_max_ns=20000, inject_start_ns=5000)],
    ids=["spec-default-fence-free", "spec-tagged", "spec-tagged-stagger", "spec-relaxed-stagger",
         "ll-stagger"])
def test_decode_allreduce_300000_epochs_soak(cfg):
    # 30 runs of 10,000 epochs on one plan (epochs 1..300,000: the 16-bit epoch fields of
    # the flag words wrap four times), every epoch of every run checked against the oracle
    R, n, pool, E, runs = 8, 4096, 7, 10000, 30
    ins, expect = _decode_case(R, n, pool, seed=21)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), **cfg)
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    for run in range(runs):
        for o in outs:
            o.fill_(-1)
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool,
                 out_epoch_stride=n * 2)
        st = plan.status()
        assert st["code"] == 0, (run, st)
        # (each run counts its inputs from the pool's first set; the flag epochs go on)
        assert _check_epochs(outs, expect, E, pool) == 0, run
    assert plan.status()["epochs"] == E * runs
    plan.free()


@pytest.mark.parametrize("check", ["tagged", "relaxed"])
def test_specialised_and_stamped_engines_agree(check):
    # a plain speculative run of the decode plan takes the variant specialised for it; with
    # one stamp per epoch it takes the specialised variant that also stamps, and with four
    # stamps per epoch the general engine: all give the oracle's bits, and the stamps
    # advance with every epoch
    R, n, pool, E = 8, 4096, 7, 1000
    ins, expect = _decode_case(R, n, pool, seed=23)
    nm = namings.allreduce(R, n, "bf16")
    got = []
    for cfg in (dict(), dict(record_stamps=1, stamp_capacity=E),
                dict(record_stamps=2, stamp_capacity=E)):
        plan = cdc.Plan(nm, protocol="spec", spec_check=check, **cfg)
        outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool,
                 out_epoch_stride=n * 2)
        assert plan.status()["code"] == 0, cfg
        assert _check_epochs(outs, expect, E, pool) == 0, cfg
        if cfg:
            per = 4 if cfg["record_stamps"] == 2 else 1
            st = plan.stamps(E).astype(np.int64)
            assert len(st) == per * E + 1
            assert (np.diff(st[1:].reshape(E, per)[:, 0]) > 0).all()
        got.append(outs)
        plan.free()
    for a, b in zip(got[0], got[1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("delay", [0, 50, 200, 2000])
@pytest.mark.parametrize("check", ["tagged", "relaxed", "literal"])
def test_speculation_delay_keeps_the_bits(check, delay):
    # the wait before the first speculative loads moves only timing: every epoch stays the
    # oracle's, on the specialised variants (tagged, relaxed) and the general engine
    R, n, pool, E = 8, 4096, 7, 2000
    ins, expect = _decode_case(R, n, pool, seed=24)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="spec", spec_check=check,
                    spec_delay_ns=delay)
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    st = plan.status()
    assert st["code"] == 0, st
    assert st["spec_checks"] == E * R * 16
    assert _check_epochs(outs, expect, E, pool) == 0
    plan.free()


def test_speculation_delay_is_validated():
    nm = namings.allreduce(2, 1024, "bf16")
    for bad in (-2, 100001):
        with pytest.raises(cdc.CollError):
            cdc.Plan(nm, protocol="spec", spec_delay_ns=bad)


@pytest.mark.parametrize("protocol", ["barrier", "dual", "spec", "ll"])
@pytest.mark.parametrize("datapath", ["oneshot", "twoshot", "twoshot_pull"])
@pytest.mark.parametrize("chain", [0, 1])
def test_decode_allreduce_epochs_bit_exact(protocol, datapath, chain):
    R, n, pool, E = 8, 4096, 7, 2000
    ins, expect = _decode_case(R, n, pool)
    nm = namings.allreduce(R, n, "bf16")
    if protocol == "ll" and datapath == "twoshot_pull":
        with pytest.raises(cdc.CollError):  # tagged data has no flags to pull on
            cdc.Plan(nm, protocol=protocol, datapath=datapath, chain=chain)
        return
    plan = cdc.Plan(nm, protocol=protocol, datapath=datapath, chain=chain)
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    st = plan.status()
    assert st["code"] == 0, st
    assert _check_epochs(outs, expect, E, pool) == 0
    # a second run continues the epoch count and stays exact
    plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    assert plan.status()["code"] == 0
    assert _check_epochs(outs, expect, E, pool) == 0
    plan.reset()
    plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    assert plan.status()["code"] == 0
    assert _check_epochs(outs, expect, E, pool) == 0
    plan.free()


@pytest.mark.parametrize("check", ["tagged", "relaxed"])
def test_chained_specialised_variants_bit_exact(check):
    # chained epochs (a rank stages epoch e + 1 only after its whole epoch-e output is done)
    # on the variants specialised for one item per warp, both speculative checks; two runs,
    # every epoch against the oracle
    R, n, pool, E = 8, 4096, 7, 5000
    ins, expect = _decode_case(R, n, pool, seed=31)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="spec", spec_check=check, chain=1)
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    for _ in range(2):
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool,
                 out_epoch_stride=n * 2)
        st = plan.status()
        assert st["code"] == 0, st
        assert _check_epochs(outs, expect, E, pool) == 0
    plan.free()


@pytest.mark.parametrize("cfg", [dict(protocol="barrier"), dict(protocol="dual"),
                                 dict(protocol="spec"), dict(protocol="spec", spec_check="relaxed"),
                                 dict(protocol="spec", spec_check="literal"),
                                 dict(protocol="dual", datapath="twoshot_pull")],
                         ids=lambda c: "-".join(str(v) for v in c.values()))
def test_flag_epochs_cross_the_16_bit_wrap(cfg):
    # producer flags keep the epoch modulo 2^16: run past epoch 65,536 (one launch, and a
    # second launch continuing the count) and check the last epochs against the oracle
    R, n, pool = 8, 1024, 7
    ins, expect = _decode_case(R, n, pool, seed=21)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), **cfg)
    tail = 64
    E1 = 65_530
    outs = [torch.zeros(tail, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    # epochs 1..E1 overwrite one scratch row each (only the flags' progress matters here)
    scratch = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, scratch, n_epochs=E1, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=0)
    assert plan.status()["code"] == 0
    # the next launch continues at epoch E1 + 1 and crosses 65,536
    E2 = tail
    plan.run(ins, outs, n_epochs=E2, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    st = plan.status()
    assert st["code"] == 0, st
    # epoch E1 + 1 + i of the plan reads pool entry i % pool of this launch
    assert _check_epochs(outs, expect, E2, pool) == 0
    plan.free()


@pytest.mark.parametrize("protocol", ["ll", "dual", "spec"])
def test_reset_then_rerun_with_new_inputs(protocol):
    # after coll_reset epochs count from 1 again: nothing left from the earlier run (flags,
    # or the epochs inside tagged-data words) may pass for the new run's
    R, n = 8, 4096
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, protocol=protocol)
    outs = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    for rep in range(3):
        rng = synth.seeded_rng(700 + rep)
        xs = [synth.normal_bf16(rng, n) for _ in range(R)]
        plan.run([to_dev(x, "bf16") for x in xs], outs)
        assert plan.status()["code"] == 0
        want = collectives.allreduce(xs, "bf16")[0]
        for o in outs:
            assert bits_equal(from_dev(o, "bf16"), want), rep
        plan.reset()
    plan.free()


def test_decode_allreduce_10000_epochs_spec_equals_barrier_under_stagger():
    R, n, pool, E = 8, 4096, 7, 10000
    ins, expect = _decode_case(R, n, pool)
    nm = namings.allreduce(R, n, "bf16")
    res = {}
    for name, cfg in [("barrier", dict(protocol="barrier")),
                      ("dual", dict(protocol="dual")),
                      ("spec", dict(protocol="spec", spec_check="tagged")),
                      ("spec-stagger", dict(protocol="spec", spec_check="tagged", inject="stagger",
                                            inject_seed=2, inject_prob_ppm=100000,
                                            inject_max_ns=20000, inject_start_ns=5000)),
                      ("spec-relaxed", dict(protocol="spec", spec_check="relaxed")),
                      ("spec-relaxed-stagger", dict(protocol="spec", spec_check="relaxed",
                                                    inject="stagger", inject_seed=3,
                                                    inject_prob_ppm=100000, inject_max_ns=20000,
                                                    inject_start_ns=5000)),
                      ("ll", dict(protocol="ll")),
                      ("ll-stagger", dict(protocol="ll", inject="stagger", inject_seed=5,
                                          inject_prob_ppm=100000, inject_max_ns=20000,
                                          inject_start_ns=5000)),
                      ("spec-twoshot-stagger", dict(protocol="spec", datapath="twoshot",
                                                    inject="stagger", inject_seed=4,
                                                    inject_prob_ppm=100000, inject_max_ns=20000)),
                      ("dual-pull-stagger", dict(protocol="dual", datapath="twoshot_pull",
                                                 inject="stagger", inject_seed=6,
                                                 inject_prob_ppm=100000, inject_max_ns=20000,
                                                 inject_start_ns=5000)),
                      ("spec-pull", dict(protocol="spec", datapath="twoshot_pull"))]:
        plan = cdc.Plan(nm, **cfg)
        outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool,
                 out_epoch_stride=n * 2)
        st = plan.status()
        assert st["code"] == 0, (name, st)
        assert _check_epochs(outs, expect, E, pool) == 0, name
        res[name] = (outs, st)
        plan.free()
    for name in res:
        for a, b in zip(res[name][0], res["barrier"][0]):
            assert torch.equal(a, b)
    assert res["spec"][1]["spec_checks"] == E * R * 16
    # the content tags of producer and consumer agree: first attempts do pass (tags computed
    # differently on the two sides would fail every one); how many pass depends on how
    # closely the warps run in step and on the speculation delay
    assert res["spec"][1]["spec_retries"] < 0.9 * res["spec"][1]["spec_checks"]
    assert res["spec-relaxed"][1]["spec_retries"] < 0.9 * res["spec-relaxed"][1]["spec_checks"]


def test_speculation_with_adversarial_pause_tagged_is_exact_literal_is_not():
    # consumer rank 2 loads its peers' payloads, signals, then pauses; rank 3 stages each
    # epoch only after that signal, inside the pause. The pages' literal flag-sum check then accepts the stale
    # payload (the falsifier of the monotonicity premise); the content tag rejects it and
    # the retry path reloads.
    R, n, pool, E = 8, 4096, 7, 300
    ins, expect = _decode_case(R, n, pool)
    nm = namings.allreduce(R, n, "bf16")
    bad = {}
    for check in ("tagged", "relaxed", "literal"):
        plan = cdc.Plan(nm, protocol="spec", spec_check=check, inject="spec_pause", inject_rank=2,
                        inject_max_ns=200000, inject_pause_ns=20000)
        outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool,
                 out_epoch_stride=n * 2)
        st = plan.status()
        assert st["code"] == 0, st
        bad[check] = (_check_epochs(outs, expect, E, pool), st["spec_retries"])
        plan.free()
    assert bad["tagged"][0] == 0
    assert bad["tagged"][1] > 0
    assert bad["relaxed"][0] == 0
    assert bad["relaxed"][1] > 0
    assert bad["literal"][0] > 0


@pytest.mark.parametrize("protocol,datapath", [("dual", "oneshot"), ("ll", "oneshot"),
                                               ("dual", "twoshot_pull")])
def test_missing_notify_times_out_and_the_gpu_stays_usable(protocol, datapath):
    R, n = 4, 1024
    rng = synth.seeded_rng(5)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, protocol=protocol, datapath=datapath, inject="skip_notify", inject_rank=1,
                    spin_limit_ns=20_000_000)
    ins = [to_dev(x, "bf16") for x in xs]
    outs = [empty_dev(n, "bf16") for _ in range(R)]
    plan.run(ins, outs, n_epochs=5)
    st = plan.status()
    assert st["code"] == cdc._lib.D["COLL_ETIMEDOUT"], st
    assert st["fail_epoch"] == 1
    plan.free()
    got, _ = run_once(nm, xs, protocol="dual")
    want = collectives.allreduce(xs, "bf16")
    assert bits_equal(got[0], want[0])


def test_bound_run_repeats_the_same_call():
    R, n = 8, 4096
    ins, expect = _decode_case(R, n, 1, seed=51)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="spec")
    outs = [torch.zeros(1, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    run = plan.bind(ins, outs)
    for _ in range(5):
        run()
    assert plan.status()["code"] == 0
    assert _check_epochs(outs, expect, 1, 1) == 0
    assert plan.status()["spec_checks"] == 5 * R * 16
    plan.free()


def test_run_rejects_aliasing_and_misalignment():
    nm = namings.allreduce(2, 1024, "bf16")
    plan = cdc.Plan(nm, protocol="spec")
    a = torch.zeros(4096, dtype=torch.int16, device="cuda")
    code = plan.run_ptrs([a.data_ptr(), a.data_ptr() + 2048], [a.data_ptr() + 2048, a.data_ptr() + 6000])
    assert code == cdc._lib.D["COLL_EOVERLAP"]
    code = plan.run_ptrs([a.data_ptr() + 2, a.data_ptr() + 4096], [a.data_ptr() + 8192 - 2048, 0])
    assert code in (cdc._lib.D["COLL_EALIGN"], cdc._lib.D["COLL_EINVAL"])
    # degenerate run arguments: no epochs, an empty input pool, a missing rank's buffer,
    # output epochs that overlap each other
    b = torch.zeros(4 * 4096, dtype=torch.int16, device="cuda")
    ins = [b.data_ptr(), b.data_ptr() + 2048]
    outs = [b.data_ptr() + 8192, b.data_ptr() + 16384]
    E = cdc._lib.D
    assert plan.run_ptrs(ins, outs, n_epochs=0) == E["COLL_EINVAL"]
    assert plan.run_ptrs(ins, outs, in_pool=0) == E["COLL_EINVAL"]
    assert plan.run_ptrs([ins[0], 0], outs) == E["COLL_EINVAL"]
    assert plan.run_ptrs(ins, outs, n_epochs=2, out_epoch_stride=1024) == E["COLL_EOVERLAP"]
    assert plan.run_ptrs(ins, outs) == 0  # and the plan still runs
    assert plan.status()["code"] == 0
    plan.free()


def test_binding_rejects_buffers_too_small_for_the_run():
    # the library sees addresses only: the binding checks each tensor's storage against the
    # bytes the run will touch (epoch strides included) before anything is enqueued
    R, n = 2, 1024
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, protocol="dual")
    E = cdc._lib.D
    ins = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    outs = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    short = [torch.zeros(n - 8, dtype=torch.int16, device="cuda"), outs[1]]
    with pytest.raises(cdc.CollError) as e:
        plan.run(ins, short)
    assert e.value.code == E["COLL_EBOUNDS"]
    with pytest.raises(cdc.CollError) as e:  # 3 epochs of output need 3 n elements
        plan.run(ins, outs, n_epochs=3, out_epoch_stride=2 * n)
    assert e.value.code == E["COLL_EBOUNDS"]
    with pytest.raises(cdc.CollError) as e:  # an input pool of 2 sets
        plan.bind(ins, outs, in_pool=2, in_epoch_stride=2 * n)
    assert e.value.code == E["COLL_EBOUNDS"]
    with pytest.raises(ValueError):
        plan.run([x.cpu() for x in ins], outs)
    # a view into a larger storage may reach beyond the view itself
    big = torch.zeros(3, n, dtype=torch.int16, device="cuda")
    plan.run(ins, [big[0], outs[1]], n_epochs=3, out_epoch_stride=0)
    plan.run(ins, [big[0, :8], big[1, :8]], n_epochs=1)  # storage covers both ranks' outputs
    assert plan.status()["code"] == 0
    plan.free()


# ------------------------------------------------------------ full-size cases

def test_prefill_allreduce_64mib_oneshot_and_twoshot_full():
    R, n = 8, 8192 * 4096
    rng = synth.seeded_rng(4)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    want = collectives.allreduce(xs, "bf16")[0]
    want_dev = to_dev(want, "bf16")
    ins = [to_dev(x, "bf16") for x in xs]
    nm = namings.allreduce(R, n, "bf16")
    for dp in ("oneshot", "twoshot"):
        plan = cdc.Plan(nm, zero_copy=1, datapath=dp)
        outs = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run(ins, outs)
        assert plan.status()["code"] == 0
        for o in outs:
            assert torch.equal(o, want_dev), dp
        plan.free()


@pytest.mark.parametrize("kind,dtype", [("reduce_scatter", "bf16"), ("reduce_to_root", "bf16"),
                                        ("reduce_scatter", "f32")])
def test_many_to_one_64mib_guided_tail_full(kind, dtype):
    # 64 MiB per rank: long enough (over 16 tiles per CTA) for the ring to claim its last
    # tiles in guided sizes; every output element against the oracle, twice (the second run
    # starts from the claim counter the first run's last CTA reset)
    R = 8
    n = (64 << 20) // (2 if dtype == "bf16" else 4)
    rng = synth.seeded_rng(3)
    gen_u = synth.uniform_bf16 if dtype == "bf16" else synth.uniform_f32
    xs = [gen_u(rng, n) for _ in range(R)]
    if kind == "reduce_scatter":
        want = collectives.reduce_scatter(xs, dtype)
    else:
        want = [collectives.allreduce(xs, dtype)[0]]
    nm = getattr(namings, kind)(R, n, dtype)
    plan = cdc.Plan(nm, zero_copy=1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.info.bulk_tile_bytes > 0 and plan.info.n_tiles >= 64 * sms
    ins = [to_dev(x, dtype) for x in xs]
    outs = [empty_dev(L, dtype) for L in nm.out_len]
    for rep in range(2):
        for o in outs:
            o.fill_(0)
        plan.run(ins, outs)
        assert plan.status()["code"] == 0
        for d, w in enumerate(want):
            assert torch.equal(outs[d].view(torch.uint8), to_dev(w, dtype).view(torch.uint8)), \
                (kind, dtype, rep, d)
    plan.free()


@pytest.mark.parametrize("kind,mib", [("broadcast", 64), ("allgather", 16), ("broadcast", 16),
                                      ("allgather", 4)])
def test_multi_destination_copies_16k_tiles_full(kind, mib):
    # jobs that write each byte to every rank run on 16 KiB tiles with up to 12 stages (the
    # 16 MiB broadcast and the 4 MiB all-gather also split each job's destinations in two);
    # every output byte against the oracle
    R, n = 8, (mib << 20) // 2
    rng = synth.seeded_rng(3)
    xs = [synth.uniform_bf16(rng, n) for _ in range(R)]
    want = collectives.broadcast(xs, 0) if kind == "broadcast" else collectives.allgather(xs)
    nm = getattr(namings, kind)(R, n, "bf16")
    plan = cdc.Plan(nm, zero_copy=1)
    assert plan.info.bulk_tile_bytes == 16384
    ins = [to_dev(x, "bf16") for x in xs]
    outs = [torch.zeros(L, dtype=torch.int16, device="cuda") for L in nm.out_len]
    plan.run(ins, outs)
    assert plan.status()["code"] == 0
    for d in range(R):
        assert torch.equal(outs[d], to_dev(want[d], "bf16")), (kind, d)
    plan.free()


@pytest.mark.parametrize("kind", ["reduce_scatter", "broadcast"])
def test_bulk_ring_back_to_back_runs_each_exact(kind):
    # 40 launches back to back (each may start while the previous one finishes), cycling two
    # input sets into distinct outputs; every output of every launch against the oracle. The
    # 16 MiB reduce-scatter claims its tail in guided sizes; the 16 MiB broadcast splits its
    # destinations over two jobs. Both issue from two producer warps.
    R, n, runs = 8, (16 << 20) // 2, 40
    rng = synth.seeded_rng(86)
    sets = [[synth.uniform_bf16(rng, n) for _ in range(R)] for _ in range(2)]
    if kind == "reduce_scatter":
        wants = [collectives.reduce_scatter(xs, "bf16") for xs in sets]
    else:
        wants = [collectives.broadcast(xs, 0) for xs in sets]
    nm = getattr(namings, kind)(R, n, "bf16")
    plan = cdc.Plan(nm, zero_copy=1)
    assert plan.info.bulk_tile_bytes > 0
    ins = [[to_dev(x, "bf16") for x in xs] for xs in sets]
    want_dev = [[to_dev(w, "bf16") for w in ws] for ws in wants]
    outs = [[torch.zeros(L, dtype=torch.int16, device="cuda") for L in nm.out_len]
            for _ in range(runs)]
    for i in range(runs):
        plan.run(ins[i % 2], outs[i])
    torch.cuda.synchronize()
    assert plan.status()["code"] == 0
    for i in range(runs):
        for d in range(R):
            assert torch.equal(outs[i][d], want_dev[i % 2][d]), (kind, i, d)
    plan.free()


def test_moe_dispatch_full_size():
    R, T, H, E, k = 8, 4096, 7168, 256, 8
    routing = synth.zipf_topk_routing(5, R, T, E, k, 1.1)
    rng = synth.seeded_rng(5)
    xs = [synth.normal_bf16(rng, (T, H)) for _ in range(R)]
    nm = namings.moe_dispatch(routing, E // R, H)
    want, counts = collectives.moe_dispatch(xs, routing, E // R)
    assert counts == nm.meta["counts"]
    plan = cdc.Plan(nm, zero_copy=1)
    ins = [to_dev(x.ravel(), "bf16") for x in xs]
    outs = [torch.empty(L, dtype=torch.int16, device="cuda") for L in nm.out_len]
    plan.run(ins, outs)
    assert plan.status()["code"] == 0
    for d in range(R):
        got = from_dev(outs[d][:counts[d] * H], "bf16")
        assert bits_equal(got, want[d].ravel())
    plan.free()


@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter", "allgather", "broadcast", "alltoall",
                                  "reduce_to_root", "gather", "scatter"])
def test_sweep_256mib_sampled(kind):
    # the largest sweep size: check 4096 sampled output elements per rank against the
    # oracle's definition evaluated at exactly those elements
    R, n = 8, (256 << 20) // 2
    ins = [synth.device_uniform_bf16(torch, 3000 + r, n, "cuda") for r in range(R)]
    nm = getattr(namings, kind)(R, n, "bf16")
    dp = "twoshot" if kind == "allreduce" else "oneshot"
    plan = cdc.Plan(nm, zero_copy=1, datapath=dp)
    outs = [torch.empty(L, dtype=torch.int16, device="cuda") for L in nm.out_len]
    plan.run(ins, outs)
    assert plan.status()["code"] == 0
    rng = synth.seeded_rng(33)
    b = n // R

    def pick(r, positions):  # input elements of rank r at the given positions
        return from_dev(ins[r][torch.from_numpy(positions).cuda()], "bf16")

    for d in range(R):
        if kind in ("reduce_to_root", "gather") and d != 0:
            continue  # only the root's output is named
        L = nm.out_len[d]
        idx = np.sort(rng.integers(0, L, 4096))
        got = from_dev(outs[d][torch.from_numpy(idx).cuda()], "bf16")
        if kind in ("allreduce", "reduce_scatter", "reduce_to_root"):
            src = idx + d * b if kind == "reduce_scatter" else idx
            want = collectives.allreduce([pick(r, src) for r in range(R)], "bf16")[0]
        elif kind in ("allgather", "gather"):
            # output element i is element i % n of rank i // n's input
            want = np.empty(idx.size, np.uint16)
            for s_ in range(R):
                m = idx // n == s_
                if m.any():
                    want[m] = pick(s_, idx[m] % n)
        elif kind == "broadcast":
            want = pick(0, idx)
        elif kind == "scatter":
            want = pick(0, idx + d * b)
        else:
            # all-to-all: block s of rank d's output is block d of rank s's input
            want = np.empty(idx.size, np.uint16)
            for s_ in range(R):
                m = idx // b == s_
                if m.any():
                    want[m] = pick(s_, d * b + idx[m] % b)
        assert bits_equal(got, want), (kind, d)
    plan.free()
    del outs, ins
    torch.cuda.empty_cache()


def test_zero_copy_plan_replays_inside_a_cuda_graph():
    R, n = 8, 1 << 16
    rng = synth.seeded_rng(81)
    xs = [synth.uniform_bf16(rng, n) for _ in range(R)]
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, zero_copy=1, datapath="twoshot")
    ins = [to_dev(x, "bf16") for x in xs]
    outs = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run(ins, outs)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    with torch.cuda.graph(g):
        plan.run(ins, outs)
    g.replay()
    torch.cuda.synchronize()
    assert plan.status()["code"] == 0
    want = collectives.allreduce(xs, "bf16")[0]
    for o in outs:
        assert bits_equal(from_dev(o, "bf16"), want)
    plan.free()


@pytest.mark.parametrize("cfg", [dict(protocol="spec"), dict(protocol="dual"),
                                 dict(protocol="barrier"), dict(protocol="spec", chain=1),
                                 dict(protocol="dual", datapath="twoshot_pull"),
                                 dict(protocol="ll"), dict(protocol="spec", spec_check="relaxed")],
                         ids=lambda c: "-".join(str(v) for v in c.values()))
def test_staged_plan_replays_inside_a_cuda_graph(cfg):
    # a captured staged run clears the plan's flags and counts its epochs from 1 on every
    # replay; new input contents between replays must show up in the outputs
    R, n, E = 8, 4096, 3
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, **cfg)
    ins = [torch.zeros(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    outs = [torch.zeros(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    kw = dict(n_epochs=E, in_epoch_stride=2 * n, in_pool=E, out_epoch_stride=2 * n)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run(ins, outs, **kw)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run(ins, outs, **kw)
    for rep in range(3):
        rng = synth.seeded_rng(600 + rep)
        xs = [[synth.normal_bf16(rng, n) for _ in range(E)] for _ in range(R)]
        for r in range(R):
            ins[r].copy_(torch.stack([to_dev(x, "bf16") for x in xs[r]]))
        g.replay()
        torch.cuda.synchronize()
        assert plan.status()["code"] == 0, rep
        for e in range(E):
            want = collectives.allreduce([xs[r][e] for r in range(R)], "bf16")[0]
            for r in range(R):
                assert bits_equal(from_dev(outs[r][e], "bf16"), want), (rep, e, r)
    # a direct run after the replays
    plan.run(ins, outs, **kw)
    assert plan.status()["code"] == 0
    for e in range(E):
        want = collectives.allreduce([xs[r][e] for r in range(R)], "bf16")[0]
        assert bits_equal(from_dev(outs[0][e], "bf16"), want)
    plan.free()


# The fused producer computes every output of y_r = W_r x_r as the plain ordered chain over
# k (one binary32 chain per output column, in row order), so its outputs equal the oracle's
# bit for bit: the rank-order sum over ranks of oracle.collectives.gemv_payloads.

def fused_sum_ok(got, wts, xs):
    """got: bf16 patterns of the rank-order sum over ranks of the payloads W_r x_r."""
    want = collectives.allreduce(collectives.gemv_payloads(wts, xs), "bf16")[0]
    return bits_equal(got, want)


def fused_epoch_expect(wts, xs_by_set):
    """Device tensor [sets, n] of the oracle's output for each input set."""
    return torch.stack([to_dev(collectives.allreduce(collectives.gemv_payloads(wts, xs),
                                                     "bf16")[0], "bf16") for xs in xs_by_set])


def test_fused_run_replays_inside_a_cuda_graph_and_follows_new_weights():
    # the weight matrices' tensor maps travel as kernel parameters: a captured fused run keeps
    # the maps it was captured with, and a direct run with other matrices (or another k)
    # re-encodes them
    R, n, k, E = 4, 2048, 256, 3
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, protocol="spec")
    rng = synth.seeded_rng(610)
    wts = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    xs_dev = [torch.zeros(E, k, dtype=torch.int16, device="cuda") for _ in range(R)]
    outs = [torch.zeros(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    kw = dict(n_epochs=E, x_epoch_stride=2 * k, x_pool=E, out_epoch_stride=2 * n)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run_gemv(dw, xs_dev, k, outs, **kw)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run_gemv(dw, xs_dev, k, outs, **kw)
    for rep in range(2):
        xs = [[synth.normal_bf16(rng, k) for _ in range(E)] for _ in range(R)]
        for r in range(R):
            xs_dev[r].copy_(torch.stack([to_dev(x, "bf16") for x in xs[r]]))
        g.replay()
        torch.cuda.synchronize()
        assert plan.status()["code"] == 0, rep
        for e in range(E):
            xe = [xs[r][e] for r in range(R)]
            for r in range(R):
                assert fused_sum_ok(from_dev(outs[r][e], "bf16"), wts, xe), (rep, e, r)
    # other matrices, then a smaller k over the same matrices' first rows
    wts2 = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    dw2 = [to_dev(w.ravel(), "bf16") for w in wts2]
    for wl, dl, kk in ((wts2, dw2, k), (wts2, dw2, 128)):
        xs = [synth.normal_bf16(rng, kk) for _ in range(R)]
        plan.run_gemv(dl, [to_dev(x, "bf16") for x in xs], kk, [o[0] for o in outs])
        assert plan.status()["code"] == 0
        for r in range(R):
            assert fused_sum_ok(from_dev(outs[r][0], "bf16"), [w[:kk] for w in wl], xs), (kk, r)
    plan.free()


@pytest.mark.parametrize("seed", range(16))
def test_bulk_ring_on_small_aligned_namings(seed):
    # force the bulk-copy (TMA) ring on small random namings (segments scaled to 16 bytes)
    op = "copy" if seed % 4 == 0 else "sum"
    dtype = "bf16" if seed % 3 else "f32"
    k = 8 if dtype == "bf16" else 4
    R = 1 + seed % 6
    rng = synth.seeded_rng(1500 + seed)
    il, i, ol, o = synth.random_naming(rng, R, 300, 4, 4, op)
    il = [x * k for x in il]
    ol = [x * k for x in ol]
    i = [(r, off * k, c * k, nmv) for (r, off, c, nmv) in i]
    o = [(r, off * k, c * k, nmv) for (r, off, c, nmv) in o]
    nm = namings.Naming(R, op, dtype, il, namings.segs(i), ol, namings.segs(o))
    xs = [gen("normal", rng, n, dtype) for n in il]
    got, init = run_once(nm, xs, zero_copy=1, tma_min_bytes=1,
                         datapath="twoshot" if seed % 2 else "oneshot")
    want = oracle_outputs(nm, xs, init)
    for g, w in zip(got, want):
        assert bits_equal(g, w)


def test_bulk_ring_epochs_over_an_input_pool():
    R, n, pool, E = 8, 3 * 4096 + 8, 3, 5
    rng = synth.seeded_rng(82)
    pool_np = [[synth.normal_bf16(rng, n) for _ in range(R)] for _ in range(pool)]
    ins = [torch.stack([to_dev(pool_np[p][r], "bf16") for p in range(pool)]).contiguous()
           for r in range(R)]
    nm = namings.allreduce(R, n, "bf16")
    for dp in ("twoshot", "oneshot"):
        plan = cdc.Plan(nm, zero_copy=1, tma_min_bytes=1, datapath=dp)
        outs = [torch.zeros(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=2 * n, in_pool=pool,
                 out_epoch_stride=2 * n)
        assert plan.status()["code"] == 0
        for e in range(E):
            want = collectives.allreduce(pool_np[e % pool], "bf16")[0]
            for r in range(R):
                assert bits_equal(from_dev(outs[r][e], "bf16"), want), (dp, e, r)
        plan.free()


def test_bulk_ring_guided_tail_across_epochs():
    # a small reduce-scatter over 80 epochs: enough tiles in all (over 16 per CTA) for the
    # ring to claim its tail in guided sizes, with claims that cross epoch boundaries
    R, n, pool, E = 8, 1 << 16, 3, 80
    rng = synth.seeded_rng(84)
    pool_np = [[synth.uniform_bf16(rng, n) for _ in range(R)] for _ in range(pool)]
    ins = [torch.stack([to_dev(pool_np[p][r], "bf16") for p in range(pool)]).contiguous()
           for r in range(R)]
    nm = namings.reduce_scatter(R, n, "bf16")
    plan = cdc.Plan(nm, zero_copy=1, tma_min_bytes=1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.info.bulk_tile_bytes > 0 and plan.info.n_tiles * E >= 64 * sms
    m = n // R
    outs = [torch.zeros(E, m, dtype=torch.int16, device="cuda") for _ in range(R)]
    wants = [collectives.reduce_scatter(pool_np[p], "bf16") for p in range(pool)]
    for rep in range(2):
        plan.run(ins, outs, n_epochs=E, in_epoch_stride=2 * n, in_pool=pool,
                 out_epoch_stride=2 * m)
        assert plan.status()["code"] == 0
        for e in range(E):
            for r in range(R):
                assert bits_equal(from_dev(outs[r][e], "bf16"), wants[e % pool][r]), (rep, e, r)
    plan.free()


def test_bulk_plan_with_misaligned_buffers_falls_back_and_stays_exact():
    R, n = 4, 1 << 20
    rng = synth.seeded_rng(83)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, zero_copy=1, datapath="twoshot")
    big_in = [torch.zeros(n + 8, dtype=torch.int16, device="cuda") for _ in range(R)]
    big_out = [torch.zeros(n + 8, dtype=torch.int16, device="cuda") for _ in range(R)]
    ins = [b[1:n + 1] for b in big_in]  # 2-byte offset: not 16-byte aligned
    outs = [b[1:n + 1] for b in big_out]
    for t, x in zip(ins, xs):
        t.copy_(to_dev(x, "bf16"))
    plan.run(ins, outs)
    assert plan.status()["code"] == 0
    want = collectives.allreduce(xs, "bf16")[0]
    for o in outs:
        assert bits_equal(from_dev(o, "bf16"), want)
    plan.free()


# ------------------------------------------------------------ next rows: more collectives

@pytest.mark.parametrize("kind", ["reduce_to_root", "gather", "scatter"])
@pytest.mark.parametrize("mode", ["zc", "staged-spec", "staged-barrier"])
def test_rooted_collectives(kind, mode):
    R, n = 8, 8192
    rng = synth.seeded_rng(90)
    xs = [synth.uniform_bf16(rng, n) for _ in range(R)]
    root = 3
    nm = getattr(namings, kind)(R, n, "bf16", root=root)
    cfg = dict(zero_copy=1) if mode == "zc" else dict(protocol=mode.split("-")[1])
    got, init = run_once(nm, xs, **cfg)
    want = getattr(collectives, kind)(*( [xs, "bf16", root] if kind == "reduce_to_root" else [xs, root]))
    for r in range(R):
        if want[r] is None:
            assert bits_equal(got[r], init[r])  # not named: untouched
        else:
            assert bits_equal(got[r][:len(want[r])], want[r])


@pytest.mark.parametrize("T,H,mode", [(256, 512, "zc"), (256, 512, "staged-spec"),
                                      (4096, 7168, "zc")])
def test_moe_combine(T, H, mode):
    R, E, k = 8, 256, 8
    routing = synth.zipf_topk_routing(6, R, T, E, k, 1.1)
    nm = namings.moe_combine(routing, E // R, H)
    rng = synth.seeded_rng(6)
    ys = [synth.normal_bf16(rng, L) for L in nm.in_len]
    counts = nm.meta["counts"]
    cfg = dict(zero_copy=1) if mode == "zc" else dict(protocol="spec")
    plan = cdc.Plan(nm, **cfg)
    ins = [to_dev(y, "bf16") for y in ys]
    outs = [torch.empty(T * H, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, outs)
    assert plan.status()["code"] == 0
    if T * H <= 256 * 512:
        want = collectives.moe_combine_sum([y.reshape(-1, H)[:c] for y, c in zip(ys, counts)],
                                           routing, E // R, "bf16")
        for s in range(R):
            assert bits_equal(from_dev(outs[s], "bf16"), want[s].ravel())
    else:
        # full size: check 64 sampled tokens per rank, each summed by the oracle's definition
        pos = np.zeros((R,), dtype=np.int64)
        dest = nm.meta["dest"]
        rowidx = {}
        for s in range(R):
            for t in range(T):
                for d in range(R):
                    if dest[s, t, d]:
                        rowidx[(s, t, d)] = pos[d]
                        pos[d] += 1
        srng = synth.seeded_rng(61)
        for s in range(R):
            for t in srng.integers(0, T, 64):
                terms = [ys[d][rowidx[(s, t, d)] * H:(rowidx[(s, t, d)] + 1) * H]
                         for d in range(R) if dest[s, t, d]]
                from oracle.arith import ordered_sum
                want = ordered_sum(terms, "bf16")
                got = from_dev(outs[s][t * H:(t + 1) * H], "bf16")
                assert bits_equal(got, want)
    plan.free()


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("kb", [8, 16, 32])
@pytest.mark.parametrize("protocol", ["barrier", "dual", "spec", "ll"])
@pytest.mark.parametrize("datapath", ["oneshot", "twoshot", "twoshot_pull"])
def test_fig15_cells_bit_exact(R, kb, protocol, datapath):
    # SiFAR's Fig. 15 grid: TP degree 2/4/8 x 8/16/32 KB payloads, every protocol
    if protocol == "ll" and datapath == "twoshot_pull":
        pytest.skip("tagged data has no flags to pull on (rejected at plan time)")
    n = kb * 1024 // 2
    pool, E = 5, 300
    ins, expect = _decode_case(R, n, pool, seed=15)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol=protocol, datapath=datapath)
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run(ins, outs, n_epochs=E, in_epoch_stride=n * 2, in_pool=pool, out_epoch_stride=n * 2)
    assert plan.status()["code"] == 0
    assert _check_epochs(outs, expect, E, pool) == 0
    plan.free()


# ------------------------------------------------------------ tolerance mode (tree order)

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_bytes,kind", [(1 << 16, "allreduce"), (1 << 23, "allreduce"),
                                          (1 << 16, "reduce_scatter"), (1 << 23, "reduce_scatter")])
def test_tree_order_sums_within_tolerance(dtype, n_bytes, kind):
    from oracle import tolerance
    R = 8
    es = 2 if dtype == "bf16" else 4
    n = n_bytes // es
    rng = synth.seeded_rng(95)
    xs = [gen("normal", rng, n, dtype) for _ in range(R)]
    nm = getattr(namings, kind)(R, n, dtype)
    for dp in ("oneshot", "twoshot"):
        got, _ = run_once(nm, xs, zero_copy=1, reduce_order="tree", datapath=dp)
        for r in range(R):
            terms = xs if kind == "allreduce" else [x[r * (n // R):(r + 1) * (n // R)] for x in xs]
            ok = tolerance.within_tolerance(got[r], terms, dtype)
            assert ok.all(), (dp, r, int((~ok).sum()))


def test_staged_plans_reject_the_tree_order():
    with pytest.raises(cdc.CollError):
        cdc.Plan(namings.allreduce(2, 1024, "bf16"), reduce_order="tree")


# ------------------------------------------------------------ fused producer (GEMV + AR)

def _gemv_case(R, n, k, pool, seed):
    rng = synth.seeded_rng(seed)
    wts = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    xs = [[synth.normal_bf16(rng, k) for _ in range(pool)] for _ in range(R)]
    return wts, xs


@pytest.mark.parametrize("protocol,datapath,chain,unit", [
    ("barrier", "oneshot", 0, 0), ("dual", "oneshot", 0, 0), ("spec", "oneshot", 0, 0),
    ("spec", "twoshot", 0, 0), ("spec", "oneshot", 1, 0), ("dual", "twoshot_pull", 1, 0),
    ("dual", "oneshot", 0, 432), ("spec", "oneshot", 1, 432), ("spec", "twoshot", 0, 432)])
def test_fused_gemv_allreduce_bit_exact(protocol, datapath, chain, unit):
    # unit 432: 19 pieces of 216 columns per rank (the last 208), 152 fused CTAs
    R, n, k, pool, E = 8, 4096, 256, 3, 24
    wts, xs = _gemv_case(R, n, k, pool, 97)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol=protocol, datapath=datapath,
                    chain=chain, unit_bytes=unit)
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [torch.stack([to_dev(x, "bf16") for x in xs[r]]).contiguous() for r in range(R)]
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs, n_epochs=E, x_epoch_stride=2 * k, x_pool=pool,
                  out_epoch_stride=2 * n)
    assert plan.status()["code"] == 0
    for e in range(E):
        xe = [xs[r][e % pool] for r in range(R)]
        for r in range(R):
            assert fused_sum_ok(from_dev(outs[r][e], "bf16"), wts, xe), (e, r)
    plan.free()


@pytest.mark.parametrize("chain", [0, 1])
def test_fused_gemv_2000_epochs_under_stagger(chain):
    # timing perturbation of the fused loop: ranks delayed at random (up to 20 us) and
    # started apart; every epoch must still equal the oracle
    R, n, k, pool, E = 8, 4096, 256, 3, 2000
    wts, xs = _gemv_case(R, n, k, pool, 97)
    want_dev = fused_epoch_expect(wts, [[xs[r][e] for r in range(R)] for e in range(pool)])
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="spec", chain=chain,
                    inject="stagger", inject_seed=7 + chain, inject_prob_ppm=100000,
                    inject_max_ns=20000, inject_start_ns=5000)
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [torch.stack([to_dev(x, "bf16") for x in xs[r]]).contiguous() for r in range(R)]
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs, n_epochs=E, x_epoch_stride=2 * k, x_pool=pool,
                  out_epoch_stride=2 * n)
    st = plan.status()
    assert st["code"] == 0, st
    assert _check_epochs(outs, want_dev, E, pool) == 0
    plan.free()


def test_fused_gemv_with_a_reduce_scatter_naming_and_bad_arguments():
    R, n, k = 4, 2048, 128
    wts, xs = _gemv_case(R, n, k, 1, 98)
    x0 = [x[0] for x in xs]
    plan = cdc.Plan(namings.reduce_scatter(R, n, "bf16"), protocol="dual")
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [to_dev(x[0], "bf16") for x in xs]
    outs = [torch.empty(n // R, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs)
    assert plan.status()["code"] == 0
    want = collectives.reduce_scatter(collectives.gemv_payloads(wts, x0), "bf16")
    for r in range(R):  # rank r holds block r of the sum
        assert bits_equal(from_dev(outs[r], "bf16"), want[r]), r
    with pytest.raises(cdc.CollError):
        plan.run_gemv(dw, dx, 12, outs)  # k not a multiple of 16
    with pytest.raises(cdc.CollError):
        plan.run_gemv(dw, dx, 8208, outs)  # x longer than the staging buffer (8192)
    zc = cdc.Plan(namings.allreduce(R, n, "bf16"), zero_copy=1)
    with pytest.raises(cdc.CollError):
        zc.run_gemv(dw, dx, k, [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)])
    plan.free()
    zc.free()



@pytest.mark.parametrize("k,n,wpr,unit", [(16, 4096, 0, 0), (80, 4096, 0, 0), (128, 4096, 0, 0),
                                          (1024, 4096, 0, 0), (512, 4096, 2, 0), (128, 1000, 0, 0),
                                          (256, 1000, 0, 0), (8192, 1024, 0, 0), (128, 4352, 1, 0),
                                          (320, 4096, 0, 0), (48, 2048, 0, 0),
                                          (512, 4096, 0, 432), (1024, 4096, 0, 432),
                                          (128, 1000, 0, 432), (384, 4096, 0, 256),
                                          (80, 1024, 0, 64)],
                         ids=["k16-one-partial-fill", "k80-full-and-partial-fill",
                              "k128-several-pieces-per-ring-lap",
                              "k1024-ring-wraps-inside-a-piece", "k512-four-pieces-per-warp",
                              "k128-ragged-last-piece", "k256-ragged-last-piece",
                              "k8192-largest-x", "k128-seventeen-pieces-per-warp",
                              "k320-a-piece-fills-the-ring", "k48-partial-fill",
                              "u432-k512-six-slot-ring", "u432-k1024-ring-wraps",
                              "u432-k128-ragged-last-piece", "u256-k384-two-warps-idle",
                              "u64-k80-sixteen-live-lanes"])
def test_fused_gemv_weight_ring_shapes(k, n, wpr, unit):
    # The weight rows stream through one ring of slots of 64 rows (one tensor copy each, 5
    # slots of 512-byte rows, 6 of 432-byte rows, 8 of smaller ones) shared by the compute
    # warps, and x through two buffers: these shapes cover a last fill only partly inside
    # the matrix (its rows past k read zeros), several pieces per ring lap, a piece longer
    # than the ring, a piece exactly as long, warps with several stage items (more than the
    # 16 whose sources are cached), the longest x, a last piece shorter than the unit, whose
    # copies read zeros past the matrix's columns, and units narrower than 512 bytes, whose
    # compute lanes past the unit's columns idle.
    R, pool, E = 4, 2, 6
    wts, xs = _gemv_case(R, n, k, pool, 99 + k + unit)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="dual", warps_per_rank=wpr,
                    unit_bytes=unit)
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [torch.stack([to_dev(x, "bf16") for x in xs[r]]).contiguous() for r in range(R)]
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs, n_epochs=E, x_epoch_stride=2 * k, x_pool=pool,
                  out_epoch_stride=2 * n)
    assert plan.status()["code"] == 0
    for e in range(E):
        xe = [xs[r][e % pool] for r in range(R)]
        for r in range(R):
            assert fused_sum_ok(from_dev(outs[r][e], "bf16"), wts, xe), (e, r)
    plan.free()


def test_fused_gemv_signed_zeros():
    # a chain starts from its first product: weights of -0 against x >= +0 give -0 payloads,
    # and the fixed-order sum of -0 over ranks stays -0; a rank with +0 payloads turns the
    # sum into +0
    R, n, k = 4, 1024, 128
    rng = synth.seeded_rng(93)
    xs = [(synth.normal_bf16(rng, k) & np.uint16(0x7FFF)).astype(np.uint16) for _ in range(R)]
    for signs in ((1, 1, 1, 1), (1, 0, 1, 1)):
        wts = [np.full((k, n), 0x8000 if sg else 0x0000, dtype=np.uint16) for sg in signs]
        want = collectives.allreduce(collectives.gemv_payloads(wts, xs), "bf16")[0]
        assert np.all(want == (0x8000 if all(signs) else 0x0000))
        plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="spec")
        outs = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
        plan.run_gemv([to_dev(w.ravel(), "bf16") for w in wts], [to_dev(x, "bf16") for x in xs],
                      k, outs)
        assert plan.status()["code"] == 0
        for r in range(R):
            assert bits_equal(from_dev(outs[r], "bf16"), want), (signs, r)
        plan.free()


@pytest.mark.parametrize("unsafe", ["weights", "x"])
def test_fused_gemv_product_overflow_keeps_the_separate_rounding(unsafe):
    # Each product is rounded to binary32 before it is added. Here one output's products are
    # -(2-2^-7)*2^127 and then 2^128, which overflows when rounded alone: multiply-then-add
    # gives +inf, where a fused multiply-add would give 2^120. The large magnitudes sit in
    # the weights, or in one epoch's x.
    R, n, k, E = 2, 256, 128, 3
    rng = synth.seeded_rng(94)
    wts = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    xs = [[synth.normal_bf16(rng, k) for _ in range(E)] for _ in range(R)]
    for r in range(R):
        wts[r][:, 0] = 0
    if unsafe == "weights":
        wts[0][0, 0], wts[0][1, 0] = 0xE07F, 0x6080    # -(2-2^-7)*2^65, 2^66
        for r in range(R):
            for e in range(E):
                xs[r][e][0] = xs[r][e][1] = 0x5E80     # 2^62
    else:
        wts[0][0, 0], wts[0][1, 0] = 0xDEFF, 0x5E80    # -(2-2^-7)*2^62, 2^62
        xs[0][1][0], xs[0][1][1] = 0x6000, 0x6080      # epoch 1: 2^65, 2^66
    want = [collectives.allreduce(collectives.gemv_payloads(wts, [xs[r][e] for r in range(R)]),
                                  "bf16")[0] for e in range(E)]
    if unsafe == "weights":
        assert all(w[0] == 0x7F80 for w in want)
    else:
        assert want[1][0] == 0x7F80 and want[0][0] != 0x7F80
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="dual")
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [torch.stack([to_dev(x, "bf16") for x in xs[r]]).contiguous() for r in range(R)]
    outs = [torch.empty(E, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs, n_epochs=E, x_epoch_stride=2 * k, x_pool=E,
                  out_epoch_stride=2 * n)
    assert plan.status()["code"] == 0
    for e in range(E):
        for r in range(R):
            assert bits_equal(from_dev(outs[r][e], "bf16"), want[e]), (e, r)
    plan.free()


def test_fused_gemv_rejects_a_plan_wider_than_the_gpu_and_keeps_the_plain_run():
    # 8 ranks x 32 KiB: 512 one-warp engine CTAs fit at once, 512 fused CTAs (one per SM) do not
    R, n, k = 8, 16384, 128
    nm = namings.allreduce(R, n, "bf16")
    plan = cdc.Plan(nm, protocol="dual")
    assert plan.info.n_warps > torch.cuda.get_device_properties(0).multi_processor_count
    wts, xs = _gemv_case(R, n, k, 1, 90)
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [to_dev(x[0], "bf16") for x in xs]
    outs = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    with pytest.raises(cdc.CollError):
        plan.run_gemv(dw, dx, k, outs)
    ys = collectives.gemv_payloads(wts, [x[0] for x in xs])
    plan.run([to_dev(y, "bf16") for y in ys], outs)
    assert plan.status()["code"] == 0
    want = collectives.allreduce(ys, "bf16")
    for r in range(R):
        assert bits_equal(from_dev(outs[r], "bf16"), want[r])
    plan.free()


def test_fused_gemv_missing_notify_times_out_and_the_gpu_stays_usable():
    # the engine warp gives up, releases the compute warps and stops the streaming warp,
    # which waits for the weight copies it issued before the CTA exits
    R, n, k = 4, 4096, 512
    wts, xs = _gemv_case(R, n, k, 1, 91)
    plan = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="dual", inject="skip_notify",
                    inject_rank=1, spin_limit_ns=20_000_000)
    dw = [to_dev(w.ravel(), "bf16") for w in wts]
    dx = [to_dev(x[0], "bf16") for x in xs]
    outs = [torch.empty(8, n, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.run_gemv(dw, dx, k, outs, n_epochs=8, out_epoch_stride=2 * n)
    st = plan.status()
    assert st["code"] == cdc._lib.D["COLL_ETIMEDOUT"], st
    assert st["fail_epoch"] == 1
    plan.free()
    ok = cdc.Plan(namings.allreduce(R, n, "bf16"), protocol="dual")
    ok.run_gemv(dw, dx, k, outs, n_epochs=8, out_epoch_stride=2 * n)
    assert ok.status()["code"] == 0
    for r in range(R):
        assert fused_sum_ok(from_dev(outs[r][7], "bf16"), wts, [x[0] for x in xs])
    ok.free()


@pytest.mark.parametrize("cfg", [dict(zero_copy=1), dict(zero_copy=1, datapath="twoshot"),
                                 dict(protocol="spec"), dict(protocol="ll"), dict(protocol="dual")],
                         ids=lambda c: "-".join(f"{k}={v}" for k, v in c.items()))
@pytest.mark.parametrize("R", [40, 64])
def test_more_than_32_ranks(R, cfg):
    n = 1024
    rng = synth.seeded_rng(99)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    got, _ = run_once(namings.allreduce(R, n, "bf16"), xs, **cfg)
    want = collectives.allreduce(xs, "bf16")[0]
    for g in got:
        assert bits_equal(g, want)
