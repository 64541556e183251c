"""CPU tests of the C ABI's host half: symbols, validation codes, plan shapes, namings.

No compute call is made (no GPU here); coll_validate runs the whole host compiler.
"""

import re

import numpy as np
import pytest

import collective_datapath_copy_gb300 as cdc
from collective_datapath_copy_gb300 import _lib, namings
from collective_datapath_copy_gb300.build import build
import oracle
from oracle import collectives, naming as onaming
from oracle.arith import NPTYPE
import synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def test_library_exports_every_declared_symbol():
    with open(_lib.HEADER) as f:
        text = f.read()
    declared = set(re.findall(r"^\s*(?:int|int64_t|const char \*)\s*(coll_\w+)\s*\(", text, re.M))
    assert {"coll_plan", "coll_run", "coll_free", "coll_status", "coll_strerror",
            "coll_validate", "coll_reset", "coll_stamps", "coll_plan_info",
            "coll_config_default"} <= declared
    h = _lib.lib()
    for name in declared:
        assert hasattr(h, name), name


def test_strerror_covers_codes():
    for name, code in _lib.D.items():
        if name.startswith("COLL_E"):
            assert _lib.lib().coll_strerror(code).decode() != "unknown error"


def _code(R, op, dtype, il, i, ol, o, **cfg):
    return cdc.validate_code(R, _lib.OP.get(op, 7), _lib.DTYPE.get(dtype, 9), il, namings.segs(i),
                             ol, namings.segs(o), **cfg)


MALFORMED = [
    # (R, op, dtype, in_len, in_segs, out_len, out_segs)
    (2, "sum", "bf16", (4, 4), [(0, 0, 4, 7), (1, 0, 4, 7)], (4, 4), [(0, 0, 4, 7), (1, 0, 4, 7)]),
    (2, "max", "bf16", (4, 4), [(0, 0, 4, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "sum", "bytes", (4, 4), [(0, 0, 4, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(2, 0, 4, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(0, 0, 0, 7)], (4, 4), []),
    (2, "sum", "bf16", (4, 4), [(0, 1, 4, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(0, 0, 4, 7)], (4, 4), [(1, 2, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(0, 0, 4, 7), (1, 0, 3, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(0, 0, 4, 7)], (4, 4), [(0, 0, 4, 8)]),
    (2, "copy", "bf16", (4, 4), [(0, 0, 4, 7), (1, 0, 4, 7)], (4, 4), [(0, 0, 4, 7)]),
    (2, "copy", "bf16", (4, 4), [(0, 0, 4, 7)], (8, 4), [(0, 0, 4, 7), (0, 3, 4, 7)]),
    (2, "copy", "bf16", (4, 4), [(0, 0, 4, 7)], (8, 4), [(0, 0, 4, 7), (0, 4, 4, 7)]),
    (2, "sum", "bf16", (4, 4), [(0, 0, 4, 7), (1, 0, 4, 7), (0, 0, 2, 9)], (4, 4), [(1, 0, 4, 7)]),
    (2, "sum", "f32", (4, 4), [], (4, 4), []),
    (1, "copy", "bytes", (5,), [(0, 0, 5, 1)], (5,), [(0, 0, 5, 1)]),
]


@pytest.mark.parametrize("case", MALFORMED)
def test_validation_codes_match_oracle(case):
    R, op, dt, il, i, ol, o = case
    want = onaming.validate(R, op, dt, list(il), i, list(ol), o)
    assert _code(R, op, dt, list(il), i, list(ol), o, zero_copy=1) == want


@pytest.mark.parametrize("seed", range(60))
def test_random_naming_codes_match_oracle(seed):
    rng = synth.seeded_rng(500 + seed)
    op = "copy" if seed % 2 else "sum"
    il, i, ol, o = synth.random_naming(rng, 1 + seed % 4, 10, 4, 3, op)
    # perturb: a random defect in about half the cases
    i, o = list(i), list(o)
    kind = seed % 6
    if kind == 1 and o:
        r, off, c, n = o[0]
        o[0] = (r, off + 100, c, n)
    elif kind == 2 and i:
        r, off, c, n = i[0]
        i[0] = (r, off, c + 1, n)
    elif kind == 3 and o:
        o.append((o[0][0], o[0][1], o[0][2], o[0][3]))
    elif kind == 4 and o:
        o.append((0, 0, 1, 999))
    R = 1 + seed % 4
    want = onaming.validate(R, op, "bf16", il, i, ol, o)
    assert _code(R, op, "bf16", il, i, ol, o, zero_copy=1) == want


def test_staged_plans_need_16_byte_alignment():
    E = _lib.D
    ok = _code(2, "sum", "bf16", [16, 16], [(0, 0, 8, 0), (1, 0, 8, 0)], [16, 16],
               [(0, 8, 8, 0), (1, 0, 8, 0)])
    assert ok == 0
    bad = _code(2, "sum", "bf16", [16, 16], [(0, 1, 8, 0), (1, 0, 8, 0)], [16, 16],
                [(0, 8, 8, 0), (1, 0, 8, 0)])
    assert bad == E["COLL_EALIGN"]
    # zero-copy plans accept any alignment
    assert _code(2, "sum", "bf16", [16, 16], [(0, 1, 8, 0), (1, 0, 8, 0)], [16, 16],
                 [(0, 8, 8, 0), (1, 0, 8, 0)], zero_copy=1) == 0


def test_bad_config_rejected():
    n = namings.allreduce(2, 256)
    with pytest.raises(cdc.CollError):
        cdc.validate(n, protocol=7)
    for bad in (100, 48, 520, 1024, -16):
        with pytest.raises(cdc.CollError):
            cdc.validate(n, unit_bytes=bad)
    # units of 64..512 bytes, multiples of 16: the 8 KiB name in ceil(8192 / u) units, each
    # staged by all 8 ranks (one warp per rank and unit)
    nm8 = namings.allreduce(8, 4096, "bf16")
    for u, units in ((0, 16), (512, 16), (432, 19), (256, 32), (64, 128)):
        info = cdc.validate(nm8, unit_bytes=u)
        assert (info.n_units, info.n_warps) == (units, 8 * units)
    with pytest.raises(cdc.CollError):
        cdc.validate(n, datapath=3)
    # the two-shot pull needs the staged exchange and flags
    with pytest.raises(cdc.CollError):
        cdc.validate(n, datapath="twoshot_pull", zero_copy=1)
    with pytest.raises(cdc.CollError):
        cdc.validate(n, datapath="twoshot_pull", protocol="ll")
    # the speculation delay: -1 (the check's default) up to 100 us
    for ok in (-1, 0, 200, 100000):
        cdc.validate(n, protocol="spec", spec_delay_ns=ok)
    for bad in (-2, 100001):
        with pytest.raises(cdc.CollError):
            cdc.validate(n, protocol="spec", spec_delay_ns=bad)


def test_default_config_is_the_fence_free_speculative_check():
    c = _lib.make_config()
    assert c.protocol == _lib.D["COLL_PROTO_SPEC"]
    assert c.spec_check == _lib.D["COLL_SPEC_TAGGED_RELAXED"]
    assert c.spec_delay_ns == -1


def test_buffer_lengths_beyond_the_limit_are_rejected():
    # byte sizes stay far from 64-bit overflow: at most 2^48 elements per rank's buffer
    E = _lib.D
    big = 1 << 48
    assert _code(2, "copy", "bf16", [big, 16], [(0, 0, 8, 0)], [16, 16], [(1, 0, 8, 0)],
                 zero_copy=1) == 0
    assert _code(2, "copy", "bf16", [big + 1, 16], [(0, 0, 8, 0)], [16, 16], [(1, 0, 8, 0)],
                 zero_copy=1) == E["COLL_EBOUNDS"]
    assert _code(2, "sum", "f32", [16, 16], [(0, 0, 8, 0)], [16, (1 << 63) + 16],
                 [(1, 0, 8, 0)], zero_copy=1) == E["COLL_EBOUNDS"]


def test_twoshot_pull_plan_shape():
    # 8 ranks x 4096 bf16: 16 units; each owner reduces 2 of them into the second exchange
    # buffer, and every rank pulls all 16: 16 pull items per rank, on 16 warps per rank
    nm = namings.allreduce(8, 4096, "bf16")
    push = cdc.validate(nm, protocol="dual", datapath="twoshot")
    pull = cdc.validate(nm, protocol="dual", datapath="twoshot_pull")
    assert pull.n_units == push.n_units == 16
    assert pull.n_warps == 128
    assert pull.xbuf_bytes == push.xbuf_bytes + 2 * 8192  # + reduced pieces, two parities
    assert pull.flag_bytes == push.flag_bytes + 16 * 2 * 4 + 16 * 8 * 4
    barrier = cdc.validate(nm, protocol="barrier", datapath="twoshot_pull")
    assert barrier.xbuf_bytes == 8 * 8192 + 8192


M = 1 << 20


@pytest.mark.parametrize("kind,min_bytes", [
    ("allreduce", lambda R, M: 2 * R * M),
    ("reduce_scatter", lambda R, M: (R + 1) * M),
    ("allgather", lambda R, M: (R + R * R) * M),
    ("broadcast", lambda R, M: (1 + R) * M),
    ("alltoall", lambda R, M: 2 * R * M),
])
def test_min_bytes_match_the_closed_forms(kind, min_bytes):
    R = 8
    n = M // 2
    nm = getattr(namings, kind)(R, n, "bf16")
    info = cdc.validate(nm, zero_copy=1)
    assert info.min_bytes == min_bytes(R, M)


def test_staged_allreduce_shape_for_decode_payload():
    # 8 ranks x 4096 bf16: 16 units of 512 B, one warp per (rank, unit); dual buffers
    nm = namings.allreduce(8, 4096, "bf16")
    info = cdc.validate(nm, protocol="spec")
    assert info.n_units == 16 and info.n_warps == 128
    assert info.xbuf_bytes == 2 * 8 * 8192
    info_b = cdc.validate(nm, protocol="barrier")
    assert info_b.xbuf_bytes == 8 * 8192


def _oracle_on(nm: namings.Naming, ins):
    outs = [np.zeros(n, dtype=NPTYPE[nm.dtype]) for n in nm.out_len]
    code = onaming.run_naming(nm.R, nm.op, nm.dtype, nm.in_len, nm.rows("in"), nm.out_len,
                              nm.rows("out"), ins, outs)
    assert code == 0
    return outs


@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_naming_builders_agree_with_direct_definitions(R):
    n = 4 * R * 3
    rng = synth.seeded_rng(40 + R)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    eq = lambda a, b: all(np.array_equal(x, y) for x, y in zip(a, b))
    assert eq(_oracle_on(namings.allreduce(R, n), xs), collectives.allreduce(xs, "bf16"))
    assert eq(_oracle_on(namings.reduce_scatter(R, n), xs), collectives.reduce_scatter(xs, "bf16"))
    assert eq(_oracle_on(namings.allgather(R, n), xs), collectives.allgather(xs))
    assert eq(_oracle_on(namings.broadcast(R, n, root=R - 1), xs), collectives.broadcast(xs, R - 1))
    assert eq(_oracle_on(namings.alltoall(R, n), xs), collectives.alltoall(xs))


def test_moe_naming_agrees_with_direct_dispatch():
    R, T, H, E, k = 4, 32, 8, 64, 8
    routing = synth.zipf_topk_routing(3, R, T, E, k, 1.1)
    rng = synth.seeded_rng(3)
    xs2 = [synth.normal_bf16(rng, (T, H)) for _ in range(R)]
    nm = namings.moe_dispatch(routing, E // R, H)
    alias = namings.alltoallv_from_routing(routing, E // R, H)
    assert np.array_equal(alias.out_segs, nm.out_segs) and np.array_equal(alias.in_segs, nm.in_segs)
    outs = _oracle_on(nm, [x.ravel() for x in xs2])
    want, counts = collectives.moe_dispatch(xs2, routing, E // R)
    assert nm.meta["counts"] == counts
    for d in range(R):
        assert np.array_equal(outs[d][:counts[d] * H], want[d].ravel())
    info = cdc.validate(nm, zero_copy=1)
    assert info.min_bytes == sum(2 * H * (1 + int(c)) for c in
                                 collectives.moe_dest_ranks(routing, E // R).sum(-1).ravel())


@pytest.mark.parametrize("R", [1, 3, 8])
def test_rooted_namings_agree_with_direct_definitions(R):
    n = 4 * R
    rng = synth.seeded_rng(70 + R)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    root = R - 1
    red = _oracle_on(namings.reduce_to_root(R, n, root=root), xs)
    assert np.array_equal(red[root], collectives.reduce_to_root(xs, "bf16", root)[root])
    g = _oracle_on(namings.gather(R, n, root=root), xs)
    assert np.array_equal(g[root], collectives.gather(xs, root)[root])
    sc = _oracle_on(namings.scatter(R, n, root=root), xs)
    for d in range(R):
        assert np.array_equal(sc[d], collectives.scatter(xs, root)[d])


def test_moe_combine_naming_agrees_with_direct_combine():
    R, T, H, E, k = 4, 24, 8, 32, 4
    routing = synth.zipf_topk_routing(8, R, T, E, k, 1.1)
    nm = namings.moe_combine(routing, E // R, H)
    rng = synth.seeded_rng(8)
    ys = [synth.normal_bf16(rng, (max(c, 1), H)) for c in nm.meta["counts"]]
    got = _oracle_on(nm, [y.ravel() for y in ys])
    want = collectives.moe_combine_sum([y[:c] for y, c in zip(ys, nm.meta["counts"])], routing,
                                       E // R, "bf16")
    for s_ in range(R):
        assert np.array_equal(got[s_], want[s_].ravel())
    info = cdc.validate(nm, zero_copy=1)
    assert info.n_names == R * T
