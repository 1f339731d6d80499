"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks the oracle against what the FreeToken article and plain
mathematics fix: hand-worked fixtures under tests/golden/, brute force on tiny
inputs, an independently written recency-list model of the LRU cache,
invariants of the residency table, dense-vs-routed MoE equivalence, and the
OCP MX v1.0 encoding tables.  A plausible slip in the oracle (a dropped term,
a wrong sign, a transposed matrix, an off-by-one in the LRU order) fails at
least one of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import ftsynth
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


# ------------------------------------------------------------------ routing

def test_route_golden():
    for c in gold("route_tiny.json")["cases"]:
        ids, w = oracle.route(np.array(c["logits"], dtype=np.float32), c["k"])
        assert ids.tolist() == c["ids"], c["why"]
        # the logits are rounded to float32, which moves the weights by ~1e-8
        np.testing.assert_allclose(w, np.array(c["w"]), rtol=2e-7, err_msg=c["why"])


def _brute_topk(row, k):
    """rank(e) = #experts strictly ahead of e by pairwise comparison."""
    E = len(row)
    rank = [sum(1 for o in range(E) if row[o] > row[e] or (row[o] == row[e] and o < e)) for e in range(E)]
    return [rank.index(j) for j in range(k)]


def test_route_brute_force_with_ties():
    rng = np.random.default_rng(1)
    for trial in range(300):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 4))
        vals = rng.choice(np.array([-1.0, -0.0, 0.0, 0.25, 0.5, 2.0], dtype=np.float32), size=(T, E))
        ids, w = oracle.route(vals, k)
        for t in range(T):
            assert ids[t].tolist() == _brute_topk(vals[t].tolist(), k)
            assert abs(w[t].sum() - 1.0) < 1e-12
            # weights follow the logit differences: w_i / w_j = exp(l_i - l_j)
            for a, b in itertools.combinations(range(k), 2):
                la, lb = float(vals[t, ids[t, a]]), float(vals[t, ids[t, b]])
                assert math.isclose(w[t, a] / w[t, b], math.exp(la - lb), rel_tol=1e-12)


def test_route_weights_invariant_to_logit_shift():
    lg = ftsynth.test_logits(3, 0, 5, 16)
    _, w0 = oracle.route(lg, 4)
    _, w1 = oracle.route(lg + np.float32(7.0), 4)
    np.testing.assert_allclose(w0, w1, rtol=1e-6)


def test_route_nan_rejected():
    lg = np.zeros((2, 4), dtype=np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.route(lg, 2)


# ------------------------------------------------------------------ q*

def _run_qstar(m, r_num, r_den):
    """q* through the cache step itself: m distinct cold misses, ample slots."""
    c = oracle.Cache(E_tot=max(m, 1), S=max(m, 1) + 4)
    ids = np.arange(m, dtype=np.int32)
    res = c.step(0, max(m, 1), ids, r_num, r_den, K_max=1000)
    assert res.counts[2] == m
    return int(res.counts[3])


def test_qstar_golden():
    for c in gold("qstar.json")["cases"]:
        assert _run_qstar(c["m"], *c["r"]) == c["qstar"], c


def test_qstar_degenerate_and_monotone():
    for m in range(0, 40):
        assert _run_qstar(m, 1, 1) == m  # BH = BP: all-fill
        assert _run_qstar(m, 0, 3) == 0
        prev = -1
        for rn in range(0, 25):
            q = _run_qstar(m, rn, 8)
            assert q >= prev and q <= m
            prev = q
            # within one half of m*r (rounding) unless clamped at m
            if q < m:
                assert abs(Fraction(q) - Fraction(m * rn, 8)) <= Fraction(1, 2)


# ------------------------------------------------------------------ LRU model

class RecencyListCache:
    """An independent statement of the shared LRU cache as a move-to-back list.

    order lists every slot from least to most recently used.  Slots touched in
    the same step share one time, so they go to the back sorted by slot index;
    never-used slots start in index order at the front.  This is the list
    form of ordering slots by (last use, slot index).
    """

    def __init__(self, E_tot, S):
        self.order = list(range(S))
        self.resident = {}  # expert -> slot
        self.holder = [None] * S

    def step(self, layer, E, ids, r, K_max, fill_order=0):
        uniq = sorted({layer * E + int(e) for e in ids})
        hits = [u for u in uniq if u in self.resident]
        misses = [u for u in uniq if u not in self.resident]
        touched = {self.resident[u] for u in hits}
        m = len(misses)
        qstar = min(m, math.floor(m * r + Fraction(1, 2)))
        untouched = [s for s in self.order if s not in touched]
        q = min(qstar, K_max, len(untouched))
        if fill_order == 0:
            fetch, cpu = misses[:q], misses[q:]
        else:  # the misses with the most routes in the step first, ties to the lower id
            routes = [layer * E + int(e) for e in ids]
            ranked = sorted(misses, key=lambda u: (-routes.count(u), u))
            fetch, cpu = sorted(ranked[:q]), sorted(ranked[q:])
        victims = untouched[:q]
        evicted = []
        for s, u in zip(victims, fetch):
            old = self.holder[s]
            evicted.append(-1 if old is None else old)
            if old is not None:
                del self.resident[old]
            self.resident[u] = s
            self.holder[s] = u
            touched.add(s)
        self.order = [s for s in self.order if s not in touched] + sorted(touched)
        slot_ids = [self.resident.get(layer * E + int(e), -1) for e in ids]
        return dict(uniq=uniq, hits=hits, fetch=fetch, victims=victims, evicted=evicted, cpu=cpu,
                    slot_ids=slot_ids, counts=[len(uniq), len(hits), m, q, m - q])


def _compare(res, ref):
    assert res.uniq.tolist() == ref["uniq"]
    assert res.counts.tolist() == ref["counts"]
    assert res.hit_list.tolist() == ref["hits"]
    assert res.fetch.tolist() == ref["fetch"]
    assert res.victims.tolist() == ref["victims"]
    assert res.evicted.tolist() == ref["evicted"]
    assert res.cpu_list.tolist() == ref["cpu"]
    assert res.slot_ids.tolist() == ref["slot_ids"]


def _clone(c):
    n = oracle.Cache(c.E_tot, c.S)
    n.slot_of[:] = c.slot_of
    n.expert_of[:] = c.expert_of
    n.last_use[:] = c.last_use
    n.now[:] = c.now
    return n


def _clone_model(mdl):
    n = RecencyListCache(0, len(mdl.holder))
    n.order = list(mdl.order)
    n.resident = dict(mdl.resident)
    n.holder = list(mdl.holder)
    return n


EXHAUSTIVE = [
    # (L, E, k, S): E_tot = L*E <= 6, S <= 3, k <= 2
    (1, 6, 1, 3),
    (2, 3, 2, 3),
    (3, 2, 1, 2),
    (2, 3, 1, 1),
]


@pytest.mark.parametrize("L,E,k,S", EXHAUSTIVE)
@pytest.mark.parametrize("r,K_max", [((1, 1), 2), ((1, 2), 2), ((1, 1), 1), ((0, 1), 2)])
def test_lru_exhaustive_replay(L, E, k, S, r, K_max):
    """Every route sequence up to length 5 (all layers, all k-subsets per step)
    against the recency-list model, step by step."""
    _exhaustive(L, E, k, S, r, K_max, 5)


@pytest.mark.parametrize("L,E,k,S", EXHAUSTIVE[:2])
def test_lru_exhaustive_replay_depth6(L, E, k, S):
    """Every route sequence up to length 6 for the two widest tiny caches."""
    _exhaustive(L, E, k, S, (1, 1), 2, 6)


def _exhaustive(L, E, k, S, r, K_max, depth):
    steps = [(l, list(c)) for l in range(L) for c in itertools.combinations(range(E), k)]
    rr = Fraction(*r)
    count = 0

    def dfs(c, mdl, d):
        nonlocal count
        if d == depth:
            return
        for layer, ids in steps:
            c2, m2 = _clone(c), _clone_model(mdl)
            res = c2.step(layer, E, np.array(ids, dtype=np.int32), r[0], r[1], K_max)
            ref = m2.step(layer, E, ids, rr, K_max)
            _compare(res, ref)
            count += 1
            dfs(c2, m2, d + 1)

    dfs(oracle.Cache(L * E, S), RecencyListCache(L * E, S), 0)
    assert count == sum(len(steps) ** i for i in range(1, depth + 1))


def test_lru_hand_trace():
    """S = 2 slots, one layer of 4 experts, k = 1, all-fill: a trace worked by hand."""
    c = oracle.Cache(4, 2)
    # step 1: e0 cold -> empty slot 0; step 2: e1 cold -> empty slot 1
    # step 3: e0 hit (slot 0 becomes most recent); step 4: e2 evicts LRU slot 1 (e1)
    # step 5: e1 evicts slot 0 (e0, used at step 3 < step 4)
    want = [([0], 0, 0, -1), ([1], 1, 1, -1), ([0], None, 0, None), ([2], 1, 1, 1), ([1], 0, 0, 0)]
    for ids, victim, slot, evicted in want:
        res = c.step(0, 4, np.array(ids, dtype=np.int32), 1, 1, 4)
        assert res.slot_ids.tolist() == [slot]
        if victim is None:
            assert res.counts.tolist() == [1, 1, 0, 0, 0]
        else:
            assert res.victims.tolist() == [victim] and res.evicted.tolist() == [evicted]


def _check_invariants(c, res, layer, E, ids, S, before_slot_of):
    now = int(c.now[0])
    resident = c.expert_of[c.expert_of >= 0]
    assert len(set(resident.tolist())) == resident.size  # no duplicate residents
    assert c.expert_of.size == S  # slot count fixed
    for s in range(S):  # mutual inverses
        if c.expert_of[s] >= 0:
            assert c.slot_of[c.expert_of[s]] == s
    for u in np.nonzero(c.slot_of >= 0)[0]:
        assert c.expert_of[c.slot_of[u]] == u
    n, h, m, q, cpu = res.counts.tolist()
    assert h + q + cpu == n
    for u in list(res.hit_list) + list(res.fetch):
        assert c.last_use[c.slot_of[u]] == now  # every hit or fill of this step is fresh
    for u in res.cpu_list:  # CPU experts do not change residency
        assert before_slot_of[u] == -1 and c.slot_of[u] == -1
    g = layer * E + np.asarray(ids)
    assert all((c.slot_of[gg] == sid) for gg, sid in zip(g, res.slot_ids))


@pytest.mark.parametrize("S,K_max,r", [(5, 3, (1, 1)), (12, 64, (1, 2)), (40, 8, (2, 1)), (3, 64, (3, 4))])
def test_lru_invariants_random(S, K_max, r):
    rng = np.random.default_rng(S * 131 + K_max)
    L, E, k, T = 3, 16, 4, 3
    c = oracle.Cache(L * E, S)
    mdl = RecencyListCache(L * E, S)
    for step in range(400):
        layer = int(rng.integers(0, L))
        ids = np.concatenate([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        before = c.slot_of.copy()
        lu_before = c.last_use.copy()
        res = c.step(layer, E, ids, r[0], r[1], K_max)
        _compare(res, mdl.step(layer, E, ids.tolist(), Fraction(*r), K_max))
        for v in res.victims:  # no victim was touched this step before the fill
            assert lu_before[v] < c.now[0]
        _check_invariants(c, res, layer, E, ids, S, before)


def test_lru_out_of_range_route_rejected():
    c = oracle.Cache(8, 2)
    with pytest.raises(oracle.OracleError):
        c.step(0, 8, np.array([8], dtype=np.int32), 1, 1, 2)


# ------------------------------------------------------------------ experts

def _bf16(vals):
    return ftsynth.f32_to_bf16(np.array(vals, dtype=np.float32))


def test_swiglu_golden_orientation():
    g = gold("swiglu_tiny.json")
    d, f = g["d"], g["f"]
    ex = np.concatenate([_bf16(g["W_gate"]).ravel(), _bf16(g["W_up"]).ravel(), _bf16(g["W_down"]).ravel()])
    for c in g["cases"]:
        y = oracle.expert_ffn(ex.view(np.uint8), 0, d, f, _bf16(c["x"]))
        np.testing.assert_allclose(y, c["y"], rtol=1e-14, atol=1e-15, err_msg=c["why"])


def test_e2m1_e8m0_tables():
    g = gold("mx_e2m1.json")
    for code, v in enumerate(g["e2m1"]):
        got = oracle.e2m1_value(code)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v)
    for e, v in g["e8m0"].items():
        assert oracle.e8m0_value(int(e)) == v
    assert math.isnan(oracle.e8m0_value(255))


def test_mxfp4_packing_and_layout():
    """d = f = 32; one scale byte per row.  Element 0 sits in the low nibble."""
    d = f = 32
    df = d * f
    codes = np.zeros(3 * df // 2, dtype=np.uint8)
    scales = np.full(3 * df // 32, 127, dtype=np.uint8)
    # gate row 0: element 0 = code 4 (2.0) low nibble, element 1 = code 2 (1.0) high nibble
    codes[0] = 0x24
    # up row 0: elements 0 and 1 = 1.0
    codes[df // 2 + 0] = 0x22
    # down row 0, column 0 = 1.0 (down block starts at 2*df/2)
    codes[2 * (df // 2) + 0] = 0x02
    # give down row 0 scale 128 (x2) to pin which scale byte belongs to it
    scales[2 * (df // 32) + 0] = 128
    ex = np.concatenate([codes, scales])
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    x0 = np.zeros(d, dtype=np.float32); x0[0] = 1.0
    x1 = np.zeros(d, dtype=np.float32); x1[1] = 1.0
    y0 = oracle.expert_ffn(ex, 1, d, f, _bf16(x0))
    y1 = oracle.expert_ffn(ex, 1, d, f, _bf16(x1))
    assert math.isclose(y0[0], 2.0 * (2.0 * sig(2.0)) * 1.0, rel_tol=1e-14)
    assert math.isclose(y1[0], 2.0 * (1.0 * sig(1.0)) * 1.0, rel_tol=1e-14)
    assert np.all(y0[1:] == 0) and np.all(y1[1:] == 0)


def _mx_fixture_expert():
    """The expert of tests/golden/mxfp4_scales.json packed in the canonical
    MXFP4 layout (written here from the layout's definition, not by the oracle)."""
    g = gold("mxfp4_scales.json")
    d, f = g["d"], g["f"]
    df = d * f
    mats = ("gate", "up", "down")
    codes = [np.zeros(df, dtype=np.uint8) for _ in mats]  # one code per element, row-major
    for name, row, col, code, _ in g["codes"]["entries"]:
        m = mats.index(name)
        cols = f if name == "down" else d
        codes[m][row * cols + col] = code
    packed = [(c[0::2] | (c[1::2] << 4)).astype(np.uint8) for c in codes]  # element 2i in the low nibble
    scales = []
    for name in mats:
        rows, cols = (d, f) if name == "down" else (f, d)
        r, grp = np.meshgrid(np.arange(rows), np.arange(cols // 32), indexing="ij")
        scales.append((g["scale_byte"]["offset"][name] + 2 * r + grp).astype(np.uint8).reshape(-1))
    ex = np.concatenate(packed + scales)
    assert ex.nbytes == ftsynth.expert_bytes(d, f, 1)
    return g, ex


def _mx_fixture_check(ffn):
    """Max relative error of ffn(ex, x) over the fixture's cases (inf if a
    zero element comes out nonzero)."""
    g, ex = _mx_fixture_expert()
    d, f = g["d"], g["f"]
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    worst = 0.0
    for c in g["cases"]:
        x = np.zeros(d, dtype=np.float32)
        x[c["x_ones"]] = 1.0
        y = ffn(ex, d, f, _bf16(x))
        want = np.zeros(d)
        for idx, a, z in c["y"]:
            want[idx] += a * sig(z)
        nz = want != 0
        if np.any(y[~nz] != 0):
            return math.inf
        worst = max(worst, float(np.max(np.abs(y[nz] - want[nz]) / np.abs(want[nz]))))
    return worst


def test_mxfp4_scale_addressing_golden():
    """Several rows per matrix hold nonzero codes, in both 32-column groups of
    a row, and every (row, group) has its own scale byte: the oracle must read
    the scale of the element's own row and group, the nibble of its own
    column, and W_down in [d, f] orientation."""
    err = _mx_fixture_check(lambda ex, d, f, x: oracle.expert_ffn(ex, 1, d, f, x))
    assert err < 1e-14, err


# Slips an MXFP4 reader could plausibly make, each planted in a private copy of
# the oracle's C source; the fixture above must reject every one of them.
_MX_SLIPS = {
    "scale from the column group alone": ("scales[idx / 32]", "scales[col / 32]"),
    "scales stored column-major": ("scales[idx / 32]", "scales[(size_t)(col / 32) * cols + row]"),
    "nibbles swapped": ("(idx & 1) ? (byte >> 4) : (byte & 15)", "(idx & 1) ? (byte & 15) : (byte >> 4)"),
    "W_down read transposed": ("return mx_elem(codes, scales, cols, row, col);",
                               "return which == 2 ? mx_elem(codes, scales, cols, col, row) "
                               ": mx_elem(codes, scales, cols, row, col);"),
    "gate and up swapped": ("const uint8_t* codes = ex + (size_t)which * (df / 2);",
                            "const uint8_t* codes = ex + (size_t)(which == 2 ? 2 : 1 - which) * (df / 2);"),
}


@pytest.mark.parametrize("slip", sorted(_MX_SLIPS))
def test_mxfp4_fixture_rejects_planted_slip(slip, tmp_path):
    import ctypes
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ftoracle.c")).read()
    old, new = _MX_SLIPS[slip]
    assert src.count(old) == 1, f"the oracle no longer contains {old!r}"
    (tmp_path / "m.c").write_text(src.replace(old, new))
    so = tmp_path / "m.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-o", str(so), str(tmp_path / "m.c"), "-lm"], check=True,
                   capture_output=True)
    lib = ctypes.CDLL(str(so))
    lib.or_expert_ffn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                  ctypes.c_void_p]
    lib.or_expert_ffn.restype = ctypes.c_int

    def ffn(ex, d, f, x):
        y = np.zeros(d)
        assert lib.or_expert_ffn(ex.ctypes.data, 1, d, f, x.ctypes.data, y.ctypes.data) == 0
        return y

    assert _mx_fixture_check(ffn) > 1e-3, f"the fixture did not catch: {slip}"


def _tiny_pool(E, d, f, dtype, seed=5):
    return ftsynth.make_pool(seed, 1, E, d, f, dtype, 0.05, threads=2)


@pytest.mark.parametrize("dtype", [0, 1])
def test_dense_equals_routed(dtype):
    E, d, f, k, T = 6, 64, 32, 2, 5
    pool = _tiny_pool(E, d, f, dtype)
    bx = ftsynth.expert_bytes(d, f, dtype)
    logits = ftsynth.test_logits(9, 0, T, E)
    ids, w = oracle.route(logits, k)
    hid = ftsynth.normal_bf16(7, 6, 0, 0, T * d).reshape(T, d)
    full, _, _ = oracle.moe_forward(pool, bx, dtype, d, f, ids, w, hid)
    gates = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            gates[t, ids[t, j]] = w[t, j]
    dense = oracle.dense_moe(pool, bx, dtype, d, f, E, gates, hid)
    np.testing.assert_allclose(full, dense, rtol=1e-12, atol=1e-14)
    # and an all-zero gate vector gives zero
    assert np.all(oracle.dense_moe(pool, bx, dtype, d, f, E, np.zeros((T, E)), hid) == 0)


def test_merge_split_sums_to_full():
    E, d, f, k, T = 8, 64, 32, 3, 7
    pool = _tiny_pool(E, d, f, 0)
    bx = ftsynth.expert_bytes(d, f, 0)
    ids, w = oracle.route(ftsynth.test_logits(4, 0, T, E), k)
    hid = ftsynth.normal_bf16(8, 6, 0, 0, T * d).reshape(T, d)
    rng = np.random.default_rng(0)
    for _ in range(5):
        sid = np.where(rng.random((T, k)) < 0.5, -1, 3).astype(np.int32)
        full, gpu, cpu = oracle.moe_forward(pool, bx, 0, d, f, ids, w, hid, slot_ids=sid)
        np.testing.assert_allclose(gpu + cpu, full, rtol=1e-12, atol=1e-14)
        # where every route of a token is on the GPU, the CPU part is exactly zero
        for t in range(T):
            if np.all(sid[t] >= 0):
                assert np.all(cpu[t] == 0)


def test_moe_forward_token_selection_matches_full_run():
    E, d, f, k, T = 4, 32, 32, 2, 6
    pool = _tiny_pool(E, d, f, 1)
    bx = ftsynth.expert_bytes(d, f, 1)
    ids, w = oracle.route(ftsynth.test_logits(2, 0, T, E), k)
    hid = ftsynth.normal_bf16(3, 6, 0, 0, T * d).reshape(T, d)
    full, _, _ = oracle.moe_forward(pool, bx, 1, d, f, ids, w, hid)
    sel = np.array([5, 0, 3], dtype=np.int32)
    part, _, _ = oracle.moe_forward(pool, bx, 1, d, f, ids, w, hid, tokens=sel)
    np.testing.assert_array_equal(part, full[sel])


def test_expert_linear_in_down_and_up():
    """y is linear in W_down and in W_up (scaling either by 2 doubles y exactly)."""
    d, f = 32, 16
    pool = _tiny_pool(1, d, f, 0)
    x = ftsynth.normal_bf16(1, 6, 0, 0, d)
    y = oracle.expert_ffn(pool, 0, d, f, x)
    for which in (1, 2):
        w = pool.view(np.uint16).copy()
        blk = w[which * d * f:(which + 1) * d * f]
        blk[:] = ftsynth.f32_to_bf16(ftsynth.bf16_to_f32(blk) * 2)
        y2 = oracle.expert_ffn(w.view(np.uint8), 0, d, f, x)
        np.testing.assert_allclose(y2, 2 * y, rtol=1e-13, atol=1e-16)


# ------------------------------------------------------------------ fill order: most-routed first

def test_fill_order_most_routed_hand_example():
    """8 experts, 4 empty slots, r = 1/2, three tokens routing [0,5], [5,7], [5,3]:
    all four experts miss, q* = floor(4/2 + 1/2) = 2.  Expert 5 has three routes
    and the others one each, so most-routed-first fills {5, 0} (the tie among
    0, 3, 7 goes to the lowest id) where ascending-id order fills {0, 3}."""
    ids = np.array([0, 5, 5, 7, 5, 3], dtype=np.int32)
    res = oracle.Cache(8, 4).step(0, 8, ids, 1, 2, 16, fill_order=1)
    assert res.counts.tolist() == [4, 0, 4, 2, 2]
    assert res.fetch.tolist() == [0, 5] and res.cpu_list.tolist() == [3, 7]
    assert res.victims.tolist() == [0, 1]
    assert res.slot_ids.tolist() == [0, 1, 1, -1, 1, -1]
    base = oracle.Cache(8, 4).step(0, 8, ids, 1, 2, 16, fill_order=0)
    assert base.fetch.tolist() == [0, 3] and base.cpu_list.tolist() == [5, 7]


@pytest.mark.parametrize("E,S,k,T,r,K_max", [(6, 3, 2, 3, (1, 2), 4), (8, 4, 2, 4, (1, 3), 2), (5, 2, 1, 4, (2, 3), 8)])
def test_fill_order_random_replay(E, S, k, T, r, K_max):
    """Multi-token steps (routes repeat, so route counts differ) against the
    recency-list model with the same fill order, 400 random steps each."""
    rng = np.random.default_rng(E * 100 + S * 10 + T)
    c, mdl = oracle.Cache(2 * E, S), RecencyListCache(2 * E, S)
    for step in range(400):
        layer = int(rng.integers(0, 2))
        ids = np.concatenate([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        res = c.step(layer, E, ids, r[0], r[1], K_max, fill_order=1)
        _compare(res, mdl.step(layer, E, ids.tolist(), Fraction(*r), K_max, fill_order=1))


# ------------------------------------------------------------------ MRU-retaining rebuild

def test_rebuild_retain_hand_example():
    """4 slots holding experts 10, 11, 12, 13 with last uses 5, 9, 9, 2 (slots
    0..3); a rebuild to 2 slots keeps the two most recent: experts 11 and 12
    (both used at 9; slot 1 before slot 2), in new slots 0 and 1."""
    c = oracle.Cache(16, 4)
    for s, (u, t) in enumerate([(10, 5), (11, 9), (12, 9), (13, 2)]):
        c.expert_of[s], c.slot_of[u], c.last_use[s] = u, s, t
    c.now[0] = 9
    n = c.rebuild_retain(2)
    assert n.expert_of.tolist() == [11, 12] and n.last_use.tolist() == [9, 9] and int(n.now[0]) == 9
    assert n.slot_of[11] == 0 and n.slot_of[12] == 1 and n.slot_of[10] == -1 and n.slot_of[13] == -1


@pytest.mark.parametrize("S,new_S", [(12, 20), (12, 12), (12, 5), (30, 1)])
def test_rebuild_retain_properties(S, new_S):
    """After random steps: the kept experts are a most-recent prefix of the
    residents (none left out is more recent than one kept), the table stays
    consistent, and -- when every resident fits -- the next step classifies
    every route exactly as without the rebuild."""
    rng = np.random.default_rng(S * 7 + new_S)
    L, E, k = 3, 10, 3
    c = oracle.Cache(L * E, S)
    for _ in range(60):
        layer = int(rng.integers(0, L))
        c.step(layer, E, rng.choice(E, size=k, replace=False).astype(np.int32), 1, 1, 64)
    n = c.rebuild_retain(new_S)
    kept = {int(u) for u in n.expert_of if u >= 0}
    res = {int(c.expert_of[s]): int(c.last_use[s]) for s in range(S) if c.expert_of[s] >= 0}
    assert len(kept) == min(len(res), new_S) and kept <= set(res)
    if kept:
        assert min(res[u] for u in kept) >= max([res[u] for u in set(res) - kept], default=-1)
    for i in range(new_S):
        if n.expert_of[i] >= 0:
            assert n.slot_of[n.expert_of[i]] == i and n.last_use[i] == res[int(n.expert_of[i])]
    assert int(np.count_nonzero(n.slot_of >= 0)) == len(kept)
    if new_S >= len(res):
        layer = 1
        ids = rng.choice(E, size=k, replace=False).astype(np.int32)
        a, b = c.step(layer, E, ids, 1, 1, 64), n.step(layer, E, ids, 1, 1, 64)
        assert a.hit_list.tolist() == b.hit_list.tolist() and a.miss_list.tolist() == b.miss_list.tolist()
