"""The C ABI without a GPU: it loads, exports every declared symbol, checks
its arguments before touching CUDA, and plans launches by pure host logic."""
import ctypes
import glob
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, ARG, ALIGN, ALIAS, WORKSPACE, CUDA, TIMEOUT, UNSUPPORTED = range(8)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ar_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ar_rmsnorm", "ar_rmsnorm_ex", "ar_rmsnorm_mapped", "ar_reduce_scatter_flat",
                 "ar_load_rmsnorm",
                 "ar_reserve_workspace", "ar_release_workspace", "ar_select_mode",
                 "ar_get_plan", "ar_strerror"):
        assert must in names


def declaration_comments():
    """{function: the comment block right before its declaration}."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        for m in re.finditer(r"/\*(?:(?!\*/).)*\*/\s*(?:#define[^\n]*\n\s*)*"
                             r"[A-Za-z_][\w\s\*]*?\b(ar_\w+)\s*\(", src, flags=re.S):
            block = m.group(0)
            out[m.group(1)] = block[block.rfind("/*"):block.find("*/", block.rfind("/*")) + 2]
    return out


def test_every_declaration_cites_a_passage_or_says_it_has_none():
    """Each entry point's comment names the page that defines what it does
    (the page's PR number), or says that no passage of the pages defines it."""
    comments = declaration_comments()
    assert set(comments) == set(declared_functions())
    missing = [name for name, text in comments.items()
               if not any(k in " ".join(text.replace("*", " ").split()) for k in (
                   "#3817", "#968", "#137643", "same passages", "Library utility",
                   "no counterpart"))]
    assert not missing, missing


def test_library_exports_every_declared_symbol(arlib):
    so = ctypes.CDLL(arlib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_version_and_strerror(arlib):
    assert arlib.ar_version() >= 100
    msgs = {arlib.ar_strerror(s) for s in range(8)}
    assert len(msgs) == 8 and all(msgs)
    assert arlib.ar_strerror(99) == "unknown status"


# Fake, never dereferenced device addresses: validation rejects these calls
# (or returns early for m = 0) before any CUDA call.
BASE = 0x7F0000000000


def call(arlib, n=2, m=4, H=1024, eps=1e-6, mode=0, parts=None, res=None, w=None, out=None,
         rout=None, sum_out=None):
    span = m * H * 2 + 4096
    parts = parts if parts is not None else [BASE + k * span for k in range(n)]
    res = BASE + 20 * span if res is None else res
    w = BASE + 21 * span if w is None else w
    out = BASE + 22 * span if out is None else out
    rout = BASE + 23 * span if rout is None else rout
    arr = (ctypes.c_void_p * max(len(parts), 1))(*parts)
    return arlib.lib().ar_rmsnorm_ex(arr, n, res, w, eps, m, H, out, rout, mode, None,
                                     sum_out, None)


def test_empty_call_is_a_noop(arlib):
    assert call(arlib, m=0) == OK


@pytest.mark.parametrize("kw,status", [
    (dict(n=0), ARG), (dict(n=17), ARG), (dict(m=-1), ARG), (dict(H=0), ARG),
    (dict(eps=-1.0), ARG), (dict(eps=float("nan")), ARG), (dict(eps=float("inf")), ARG),
    (dict(mode=3), ARG), (dict(H=1020), ALIGN), (dict(H=131072 + 8), UNSUPPORTED),
])
def test_bad_shapes(arlib, kw, status):
    assert call(arlib, **kw) == status


def test_null_and_misaligned_pointers(arlib):
    assert call(arlib, res=0) == ARG
    assert call(arlib, parts=[BASE, 0]) == ARG
    assert call(arlib, out=BASE + 22 * (4 * 1024 * 2 + 4096) + 8) == ALIGN
    assert call(arlib, parts=[BASE + 2, BASE + 100000]) == ALIGN
    assert call(arlib, sum_out=BASE + 30 * 100000 + 4) == ALIGN


def test_empty_call_needs_no_pointers(arlib):
    assert call(arlib, m=0, res=0, out=0, rout=0, parts=[0, 0]) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_in_place_residual_passes_the_checks(arlib):
    # Without a device the call gets past every argument check and stops at
    # the first CUDA call: AR_ERR_CUDA, not AR_ERR_ALIAS.
    span = 4 * 1024 * 2 + 4096
    res = BASE + 20 * span
    assert call(arlib, res=res, rout=res) == CUDA


def test_aliasing_rules(arlib):
    span = 4 * 1024 * 2 + 4096
    res = BASE + 20 * span
    # everything that overlaps, other than residual_out == residual, is refused
    assert call(arlib, out=res) == ALIAS
    assert call(arlib, rout=res + 16) == ALIAS
    assert call(arlib, out=BASE) == ALIAS                       # out over partial 0
    assert call(arlib, rout=BASE + span + 64) == ALIAS          # residual_out inside partial 1
    assert call(arlib, out=BASE + 30 * span, rout=BASE + 30 * span + 1024) == ALIAS
    assert call(arlib, sum_out=res) == ALIAS


def test_stage_entry_points_check_arguments(arlib):
    L = arlib.lib()
    arr = (ctypes.c_void_p * 2)(BASE, BASE + (1 << 20))
    assert L.ar_reduce_scatter_flat(arr, 2, 12, BASE + (4 << 20), None) == ALIGN
    assert L.ar_reduce_scatter_flat(arr, 0, 16, BASE + (4 << 20), None) == ARG
    assert L.ar_reduce_scatter_flat(arr, 2, 16, BASE, None) == ALIAS
    assert L.ar_reduce_scatter_flat(arr, 2, 0, BASE + (4 << 20), None) == OK
    assert L.ar_load_rmsnorm(BASE, BASE + 4096, BASE + 8192, 1e-6, 0, 1024, BASE + 12288,
                             BASE + 16384, None) == OK
    assert L.ar_load_rmsnorm(BASE, BASE + 4096, BASE + 8192, -1.0, 1, 1024, BASE + 12288,
                             BASE + 16384, None) == ARG


def test_static_scratch_entry_point_checks_shape_first(arlib):
    """ar_rmsnorm_two_stage_static runs ar_rmsnorm's shape checks in the same
    order before its own size limit, and only then treats m == 0 as a no-op
    (all of it before any CUDA call)."""
    L = arlib.lib()
    arr = (ctypes.c_void_p * 2)(BASE, BASE + (1 << 20))
    SCRATCH_LIMIT = 8
    limit = arlib.AR_STATIC_SCRATCH_ELEMS

    def call(n=2, m=4, H=1024, eps=1e-6):
        return L.ar_rmsnorm_two_stage_static(arr, n, None, None, eps, m, H, None, None, None)

    assert call(m=0, eps=float("nan")) == ARG
    assert call(m=0, eps=-1.0) == ARG
    assert call(m=0, H=1020) == ALIGN
    assert call(m=0, H=arlib.AR_MAX_HIDDEN + 8) == UNSUPPORTED
    assert call(m=0, n=0) == ARG and call(m=-1) == ARG and call(H=0) == ARG
    assert call(m=limit // 1024 + 1, H=1020) == ALIGN              # alignment before the limit
    assert call(m=limit // 8192 + 1, H=8192) == SCRATCH_LIMIT
    assert call(m=limit // 8192 + 1, H=8192, eps=float("inf")) == ARG
    assert call(m=0) == OK                                         # no pointers needed
    # ar_rmsnorm gives the same codes for the same shape errors
    for kw in (dict(m=0, eps=float("nan")), dict(m=0, H=1020), dict(m=0, H=arlib.AR_MAX_HIDDEN + 8)):
        a = {**dict(n=2, m=4, H=1024, eps=1e-6), **kw}
        assert L.ar_rmsnorm(arr, a["n"], None, None, a["eps"], a["m"], a["H"], None, None, 2,
                            None) == call(**a)


def test_cross_rank_calls_check_arguments_first(arlib):
    """The signal, barrier, two-shot, one-shot and IPC calls refuse bad
    arguments before any CUDA call."""
    L = arlib.lib()
    pads = (ctypes.c_void_p * 2)(BASE, BASE + 4096)
    assert L.ar_signal_post(pads, 0, 0, 1, None) == ARG          # world
    assert L.ar_signal_post(pads, 2, 2, 1, None) == ARG          # rank >= world
    assert L.ar_signal_post(pads, 17, 0, 1, None) == ARG
    assert L.ar_signal_post(None, 2, 0, 1, None) == ARG
    assert L.ar_signal_post((ctypes.c_void_p * 2)(BASE, 0), 2, 0, 1, None) == ARG
    assert L.ar_signal_post((ctypes.c_void_p * 2)(BASE, BASE + 4), 2, 0, 1, None) == ALIGN
    assert L.ar_signal_wait(None, 2, 1, 1000, None) == ARG
    assert L.ar_signal_wait(BASE + 4, 2, 1, 1000, None) == ALIGN
    assert L.ar_signal_wait(BASE, 2, 1, 0, None) == ARG          # unbounded wait refused
    assert L.ar_signal_wait(BASE, 2, 1, 10_000_001, None) == ARG
    assert L.ar_barrier(pads, 2, 0, 1, 0, None) == ARG
    assert L.ar_barrier(pads, 2, -1, 1, 1000, None) == ARG
    temps = (ctypes.c_void_p * 2)(BASE + (8 << 20), BASE + (12 << 20))
    parts = (ctypes.c_void_p * 2)(BASE + (16 << 20), BASE + (20 << 20))
    two_shot = lambda **k: L.ar_rmsnorm_two_shot(
        parts, 2, BASE + (24 << 20), BASE + (28 << 20), k.get("eps", 1e-6), k.get("m", 4),
        k.get("H", 1024), BASE + (32 << 20), BASE + (36 << 20), k.get("rank", 0),
        k.get("world", 2), k.get("temps", temps), k.get("pads", pads), 1, k.get("limit", 1000), None)
    assert two_shot(m=0) == OK                                     # checks only the sizes
    assert two_shot(eps=-1.0) == ARG and two_shot(H=1020) == ALIGN
    assert two_shot(rank=2) == ARG and two_shot(limit=0) == ARG
    assert two_shot(temps=(ctypes.c_void_p * 2)(BASE + (8 << 20), BASE + (8 << 20) + 8)) == ALIGN
    assert two_shot(temps=(ctypes.c_void_p * 2)(BASE + (8 << 20), BASE + (8 << 20) + 16)) == ALIAS
    assert two_shot(temps=(ctypes.c_void_p * 2)(BASE + (8 << 20), BASE + (16 << 20))) == ALIAS
    one_shot = lambda **k: L.ar_rmsnorm_one_shot(
        parts, 2, BASE + (24 << 20), BASE + (28 << 20), k.get("eps", 1e-6), k.get("m", 4),
        k.get("H", 1024), k.get("out", BASE + (32 << 20)), BASE + (36 << 20), k.get("rank", 0),
        k.get("world", 2), k.get("pads", pads), 1, k.get("limit", 1000), k.get("end", 1), None)
    assert one_shot(m=0) == OK and one_shot(m=0, end=0) == OK     # checks only the sizes
    assert one_shot(eps=float("nan")) == ARG and one_shot(H=1020) == ALIGN
    assert one_shot(rank=2) == ARG and one_shot(world=17) == ARG and one_shot(limit=0) == ARG
    assert one_shot(end=2) == ARG and one_shot(end=-1) == ARG
    assert one_shot(pads=(ctypes.c_void_p * 2)(BASE, BASE + 8)) == ALIGN
    assert one_shot(out=BASE + (16 << 20)) == ALIAS               # out on a partial
    h = ctypes.create_string_buffer(64)
    off = ctypes.c_int64(0)
    assert L.ar_ipc_get_handle(None, h, ctypes.byref(off)) == ARG
    assert L.ar_ipc_get_handle(BASE, None, ctypes.byref(off)) == ARG
    p = ctypes.c_void_p()
    assert L.ar_ipc_open(None, 0, ctypes.byref(p)) == ARG
    assert L.ar_ipc_open(h, -1, ctypes.byref(p)) == ARG
    assert L.ar_ipc_close(h) == ARG                                # never opened
    m = ctypes.c_int(0)
    assert L.ar_selftest_barrier(0, 0, 10, 1000, ctypes.byref(m)) == ARG
    assert L.ar_selftest_barrier(0, 17, 10, 1000, ctypes.byref(m)) == ARG
    assert L.ar_selftest_barrier(0, 2, 0, 1000, ctypes.byref(m)) == ARG
    assert L.ar_selftest_barrier(0, 2, 10, 0, ctypes.byref(m)) == ARG


def test_mapped_entry_point_checks_arguments_before_touching_memory(arlib):
    """ar_rmsnorm_mapped runs the same shape, alignment and alias checks as
    ar_rmsnorm before its per-pointer memory-type checks; on a machine
    without a GPU those report AR_ERR_CUDA, never a launch."""
    L = arlib.lib()
    arr = (ctypes.c_void_p * 2)(BASE, BASE + (1 << 20))
    f = ctypes.c_float
    call = lambda n, m, H, out, rout, eps=1e-6: L.ar_rmsnorm_mapped(
        arr, n, BASE + (2 << 20), BASE + (3 << 20), f(eps), m, H, out, rout, 1, None)
    assert call(0, 4, 1024, BASE + (4 << 20), BASE + (5 << 20)) == ARG
    assert call(2, 4, 1020, BASE + (4 << 20), BASE + (5 << 20)) == ALIGN
    assert call(2, 4, 1024, BASE + (4 << 20), BASE + (5 << 20), eps=-1.0) == ARG
    assert call(2, 4, 1024, BASE, BASE + (5 << 20)) == ALIAS
    assert call(2, 0, 1024, None, None) == OK
    assert call(2, 4, 1024, BASE + (4 << 20) + 8, BASE + (5 << 20)) == ALIGN
    assert call(2, 4, 1024, BASE + (4 << 20), BASE + (5 << 20)) == arlib.AR_ERR_CUDA


def test_select_mode_is_host_logic(arlib):
    for n in (1, 2, 4, 8, 16):
        for m in (1, 16, 32, 1024, 16384):
            assert arlib.ar_select_mode(n, m, 7168) in (1, 2)
    with pytest.raises(arlib.ArError):
        arlib.ar_select_mode(0, 1, 1024)


SHAPES = [(2, 4, 1024), (8, 1, 7168), (8, 16, 7168), (4, 32, 7168), (4, 2048, 7168),
          (8, 8192, 6144), (4, 1, 4096), (8, 16384, 8192), (1, 3, 8), (16, 5, 131072),
          (3, 1000, 65536), (8, 151, 7168), (8, 152, 7168), (8, 304, 7168)]


def _check_plan(p, n, m, H, mode):
    """What every plan must satisfy, whatever the table chose."""
    P = H // 8
    assert p["mode"] in (1, 2) and (mode == 0 or p["mode"] == mode)
    assert p["launches"] == (2 if p["mode"] == 2 else 1)
    assert p["vpt"] in (1, 2, 4, 8)
    # L2 prefetch: every kernel prefetches its first row before the wait on the
    # previous grid; a register kernel with one CTA per row may also prefetch
    # the row one wave ahead
    assert p["prefetch"] in ((2,) if p["kernel"] == 2 else (2, 3) if p["cluster"] == 1 else (2,))
    if p["kernel"] in (1, 3):   # register kernel: one CTA or a cluster per row
        per_cta = -(-P // p["cluster"])
        assert p["cluster"] in (1, 2, 4, 8, 16) and p["stages"] == 0
        assert p["kernel"] == 1 or p["cluster"] == 1              # late weight: one CTA per row
        assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 1024 // p["vpt"]
        assert p["threads"] * p["vpt"] >= per_cta          # every pack has an owner
        assert per_cta <= 1024                             # a row slice fits in registers
        assert p["ctas"] == m * p["cluster"]
    else:                  # stream kernel: persistent, producer warp + consumers
        assert p["kernel"] == 2 and p["cluster"] == 1
        tc = p["threads"] - 32
        assert tc % 32 == 0 and 32 <= tc <= 512
        tiles = -(-P // tc)
        assert tiles <= p["vpt"]                           # the template holds every tile
        inputs = n if p["mode"] == 1 else 1
        smem = p["stages"] * (inputs + 1) * tc * 16 + 16 * p["stages"] + 256 + 16
        per_sm = -(-p["ctas"] // 152)
        assert 2 <= p["stages"] <= 16 and per_sm * (smem + 1024) <= 233472
        assert p["ctas"] in (min(m, 152), min(m, 304))


@pytest.mark.parametrize("n,m,H", SHAPES)
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_plan_covers_every_pack(arlib, n, m, H, mode):
    _check_plan(arlib.ar_get_plan(n, m, H, mode, sm_count=152), n, m, H, mode)


def test_every_table_cell_plans_a_launchable_shape(arlib):
    """At every grid point of the plan table, and half-way between rows
    columns, both modes give a plan that satisfies the launch constraints."""
    grid, sms, _ = plan_table()
    rows = grid["kPlanRows"]
    between = [(a + b) // 2 for a, b in zip(rows, rows[1:])]
    for n in grid["kPlanInputs"]:
        for P in grid["kPlanPacks"]:
            for m in rows + between:
                for mode in (1, 2):
                    _check_plan(arlib.ar_get_plan(n, m, 8 * P, mode, sm_count=sms), n, m, 8 * P,
                                mode)


def test_plan_spreads_small_batches(arlib):
    # decode: a row of H = 7168 spreads over an 8-CTA cluster below 64 rows
    for m in (1, 4, 16, 32, 63):
        assert arlib.ar_get_plan(8, m, 7168, 1, sm_count=152)["cluster"] == 8
    assert arlib.ar_get_plan(4, 64, 7168, 1, sm_count=152)["cluster"] == 1
    # prefill: one 768-thread CTA per row, one pack per thread; with the L2
    # prefetch one wave ahead it outran the persistent stream kernel (7.2 vs
    # 7.07 TB/s), so the measured table picks it
    p = arlib.ar_get_plan(8, 8192, 6144, 1, sm_count=152)
    assert p["kernel"] == 1 and p["vpt"] == 1 and p["threads"] == 768 and p["cluster"] == 1
    assert p["ctas"] == 8192 and p["prefetch"] in (2, 3)
    # 8 inputs, H = 8192, 1024 rows: two persistent streaming CTAs per SM,
    # each with a 2-slot ring of 9 x 4 KB tiles (144 KB in flight per SM)
    p = arlib.ar_get_plan(8, 1024, 8192, 1, sm_count=152)
    assert p["kernel"] == 2 and p["ctas"] == 304 and p["stages"] == 2 and p["threads"] == 288
    # 8 inputs, H = 8192, 512 rows: the register kernel with the weight loaded
    # after the sums, two packs per thread
    p = arlib.ar_get_plan(8, 512, 8192, 1, sm_count=152)
    assert p["kernel"] == 3 and p["vpt"] == 2 and p["threads"] == 512 and p["cluster"] == 1
    # 16 inputs: one CTA per SM, 2 slots
    p = arlib.ar_get_plan(16, 8192, 6144, 1, sm_count=152)
    assert p["kernel"] == 2 and p["ctas"] == 152 and p["stages"] == 2
    # 3 inputs: the register kernel
    assert arlib.ar_get_plan(3, 8192, 4096, 1, sm_count=152)["kernel"] == 1
    # stage 2 of two-stage (one input) stays on the register kernel
    assert arlib.ar_get_plan(8, 8192, 6144, 2, sm_count=152)["kernel"] == 1
    # H above the stream kernel's limit: the register kernel with a cluster
    p = arlib.ar_get_plan(3, 1000, 65536, 1, sm_count=152)
    assert p["kernel"] == 1 and p["cluster"] == 8
    # rows of 1536 and 2048 packs (H = 12288, 16384) are in the measured table:
    # the register kernel over a 2-CTA cluster per row, or the stream kernel
    p = arlib.ar_get_plan(8, 256, 16384, 1, sm_count=152)
    assert p["kernel"] == 1 and p["cluster"] == 2 and p["vpt"] == 2
    assert arlib.ar_get_plan(8, 16384, 16384, 1, sm_count=152)["kernel"] == 2
    # rows beyond the table (more than 2048 packs): stream for >= 5 inputs
    # from 256 rows, for 4 inputs from max(4 x SMs, 1024) rows
    assert arlib.ar_get_plan(8, 255, 24576, 1, sm_count=152)["kernel"] == 1
    assert arlib.ar_get_plan(8, 256, 24576, 1, sm_count=152)["kernel"] == 2
    assert arlib.ar_get_plan(4, 1023, 24576, 1, sm_count=152)["kernel"] == 1
    assert arlib.ar_get_plan(4, 1024, 24576, 1, sm_count=152)["kernel"] == 2
    assert arlib.ar_get_plan(4, 1215, 24576, 1, sm_count=304)["kernel"] == 1


def plan_table():
    """The launch plan's lookup table, parsed from its generated header:
    (grid, SM count, score[inputs][packs][rows] = percentages per candidate)."""
    text = open(os.path.join(ROOT, "allreduce_sum_residual_gb300", "csrc", "plan_table.cuh")).read()
    grid = {name: [int(x) for x in re.search(name + r"\[\d+\] = \{([^}]*)\}", text).group(1).split(",")]
            for name in ("kPlanInputs", "kPlanPacks", "kPlanRows")}
    sms = int(re.search(r"kPlanTableSms = (\d+)", text).group(1))
    body = text[text.index("kPlanScore["):]
    ncand = int(re.search(r"kPlanCandidates = (\d+)", text).group(1))
    cells = [[int(x) for x in c.split(",")]
             for c in re.findall(r"\{(\d+(?:,\d+){%d})\}" % (ncand - 1), body)]
    ni, npk, nr = (len(grid[k]) for k in ("kPlanInputs", "kPlanPacks", "kPlanRows"))
    assert len(cells) == ni * npk * nr
    score = [[[cells[(i * npk + j) * nr + k] for k in range(nr)] for j in range(npk)] for i in range(ni)]
    return grid, sms, score


def _bracket(g, x):
    if x <= g[0]:
        return 0, 0
    for i, v in enumerate(g):
        if x == v:
            return i, i
        if x < v:
            return i - 1, i
    return len(g) - 1, len(g) - 1


def _table_pick(grid, sms_table, score, n, m, P, sms):
    """The lookup restated: bracketing inputs, packs and rows columns,
    highest summed percentage (first on ties)."""
    n0, n1 = _bracket(grid["kPlanInputs"], n)
    p0, p1 = _bracket(grid["kPlanPacks"], P)
    m0, m1 = _bracket(grid["kPlanRows"], m * sms_table / sms)
    nc = len(score[0][0][0])
    tot = [0] * nc
    for i in range(n0, n1 + 1):
        for j in range(p0, p1 + 1):
            for k in range(m0, m1 + 1):
                for c in range(nc):
                    tot[c] += score[i][j][k][c]
    return _cand_char(max(range(nc), key=lambda c: (tot[c], -c)))


def _cand_char(c):
    """Candidate index -> the header's winner character."""
    return "S1248abcd"[c]


def _expect(p, ch, P=None):
    """The plan realises the table's candidate `ch`; rows of more than 1024
    packs are split over the fewest CTAs that hold them (a cluster)."""
    cluster = 1 if P is None or P <= 1024 else -(-P // 1024)
    cluster = 1 << (cluster - 1).bit_length() if cluster > 1 else 1
    if ch == "S":
        return p["kernel"] == 2
    if ch in "abcd":
        return p["kernel"] == 3 and p["cluster"] == 1 and p["vpt"] == 1 << "abcd".index(ch)
    return p["kernel"] == 1 and p["cluster"] == cluster and p["vpt"] == int(ch)


def test_plan_follows_the_measured_table_at_every_grid_point(arlib):
    grid, sms, score = plan_table()
    for i, n in enumerate(grid["kPlanInputs"]):
        for j, P in enumerate(grid["kPlanPacks"]):
            for k, m in enumerate(grid["kPlanRows"]):
                s = score[i][j][k]
                ch = _cand_char(max(range(len(s)), key=lambda c: (s[c], -c)))
                p = arlib.ar_get_plan(n, m, 8 * P, 1, sm_count=sms)
                assert _expect(p, ch, P), (n, P, m, ch, p)


def test_plan_between_grid_points(arlib):
    """Random shapes off the grid: the plan equals the restated lookup
    (bracketing columns, SM scaling, shortest-column clamp, the one-input
    row for stage 2 of two-stage)."""
    import random
    grid, sms, score = plan_table()
    rng = random.Random(7)
    for _ in range(3000):
        n = rng.randint(1, 16)
        H = 8 * rng.randint(4, grid["kPlanPacks"][-1])
        m = int(round(10 ** rng.uniform(1.8, 4.6)))
        sm = rng.choice((sms, sms // 2, 132, 160))
        mode = rng.choice((1, 1, 1, 2))
        p = arlib.ar_get_plan(n, m, H, mode, sm_count=sm)
        inputs = n if mode == 1 else 1
        if m < 64:
            assert p["kernel"] == 1 and p["cluster"] >= 1
            continue
        ch = _table_pick(grid, sms, score, inputs, m, H // 8, sm)
        assert _expect(p, ch, H // 8), (n, m, H, mode, sm, ch, p)


def _table_pick_waves(grid, sms_table, score, n, m, P, sms, occ):
    """The wave-aware lookup restated: per candidate, a register kernel's
    rows columns are narrowed to those in the shape's own wave count (waves
    of occ(...) x the table's SMs, rows scaled to the table's SMs); the best
    mean percentage wins (first on ties)."""
    import math
    n0, n1 = _bracket(grid["kPlanInputs"], n)
    p0, p1 = _bracket(grid["kPlanPacks"], P)
    rows = m * sms_table / sms
    m0, m1 = _bracket(grid["kPlanRows"], rows)
    nc = len(score[0][0][0])
    best, best_mean = 0, -1.0
    for c in range(nc):
        lo, hi = m0, m1
        if c > 0 and m0 != m1 and P <= 1024:
            vpt = 1 << ((c - 1) % 4)
            late = 1 if c >= 5 else 0
            threads = -(-(-(-P // vpt)) // 32) * 32
            k = occ(n, vpt, late, threads)
            if k > 0:
                wave = k * sms_table
                w = math.ceil(rows / wave)
                at_lo = math.ceil(grid["kPlanRows"][m0] / wave) == w
                at_hi = math.ceil(grid["kPlanRows"][m1] / wave) == w
                if at_lo and not at_hi:
                    hi = m0
                if at_hi and not at_lo:
                    lo = m1
        vals = [score[i][j][k2][c] for i in range(n0, n1 + 1) for j in range(p0, p1 + 1)
                for k2 in range(lo, hi + 1)]
        mean = sum(vals) / len(vals)
        if mean > best_mean:
            best, best_mean = c, mean
    return _cand_char(best)


def test_wave_aware_plan_with_given_occupancy(arlib):
    """ar_get_plan_ex with a fake occupancy (CTAs per SM from a made-up
    register count per (inputs, vpt, late)) equals the restated wave-aware
    lookup on random shapes; without occupancy it is ar_get_plan."""
    import random
    grid, sms, score = plan_table()

    def occ(inputs, vpt, late, threads):
        regs = 24 + 4 * inputs * vpt - (4 * vpt if late else 0)
        regs = (min(regs, 255) + 7) // 8 * 8
        return max(1, min(65536 // (threads * regs), 2048 // threads, 32))

    rng = random.Random(11)
    differ = 0
    for _ in range(2000):
        n = rng.randint(1, 16)
        H = 8 * rng.randint(4, grid["kPlanPacks"][-1])
        m = int(round(10 ** rng.uniform(1.81, 4.4)))
        sm = rng.choice((sms, 132, 160))
        p = arlib.ar_get_plan_ex(n, m, H, 1, sm, occ)
        ch = _table_pick_waves(grid, sms, score, n, m, H // 8, sm, occ)
        assert _expect(p, ch, H // 8), (n, m, H, sm, ch, p)
        plain = arlib.ar_get_plan_ex(n, m, H, 1, sm, None)
        assert plain == arlib.ar_get_plan(n, m, H, 1, sm_count=sm)
        differ += plain != p
    assert differ > 0   # the waves do change some choices
    with pytest.raises(arlib.ArError):
        arlib.ar_get_plan_ex(4, 100, 4096, 1, 0, occ)


def test_device_occupancy_is_unknown_without_a_ready_device(arlib):
    """ar_register_occupancy reads the table a launching call fills; before
    that (here: no GPU at all) it is 0, and planning with it is the plain
    interpolation."""
    L = arlib.lib()
    assert L.ar_register_occupancy(4, 1, 0, 512) == 0
    assert L.ar_register_occupancy(0, 1, 0, 512) == 0 and L.ar_register_occupancy(4, 3, 0, 512) == 0
    for n, m, H in ((4, 300, 7168), (8, 8192, 6144), (2, 1000, 2880)):
        assert arlib.ar_get_plan_ex(n, m, H, 1, 152, L.ar_register_occupancy) == \
            arlib.ar_get_plan(n, m, H, 1, sm_count=152)
    assert L.ar_checks_bounds() == 0


def test_plan_rejects_bad_shapes(arlib):
    with pytest.raises(arlib.ArError):
        arlib.ar_get_plan(8, 4, 1020, 1, sm_count=152)
    with pytest.raises(arlib.ArError):
        arlib.ar_get_plan(8, 4, 1024, 7, sm_count=152)


def test_reduce_scatter_store_checks_arguments(arlib):
    L = arlib.lib()
    P = (ctypes.c_void_p * 2)(BASE, BASE + (1 << 20))
    T = (ctypes.c_void_p * 4)(BASE + (4 << 20), BASE + (5 << 20), BASE + (6 << 20), BASE + (7 << 20))
    call = L.ar_reduce_scatter_store
    assert call(P, 2, 1024, 0, 0, T, None) == ARG          # world 0
    assert call(P, 2, 1024, 4, 4, T, None) == ARG          # rank == world
    assert call(P, 2, 1024, -1, 4, T, None) == ARG
    assert call(P, 2, 1024, 0, 17, T, None) == ARG
    assert call(P, 2, 1020, 0, 4, T, None) == ALIGN        # count % 8
    assert call(P, 2, 0, 0, 4, None, None) == OK           # empty call needs no pointers
    Tover = (ctypes.c_void_p * 2)(BASE + (4 << 20), BASE + (4 << 20) + 512)
    assert call(P, 2, 1024, 0, 2, Tover, None) == ALIAS    # temps overlap each other
    Tpart = (ctypes.c_void_p * 2)(BASE + 64, BASE + (5 << 20))
    assert call(P, 2, 1024, 0, 2, Tpart, None) == ALIAS    # a temp overlaps a partial
    Tmis = (ctypes.c_void_p * 2)(BASE + (4 << 20) + 8, BASE + (5 << 20))
    assert call(P, 2, 1024, 0, 2, Tmis, None) == ALIGN
    # one pack spread over 4 ranks: ranks 1..3 have empty slices and launch nothing
    for r in (1, 2, 3):
        assert call(P, 2, 8, r, 4, T, None) == OK


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No CPU or torch fallback: with the shared library missing, the first
    call raises instead of computing anything."""
    code = ("import allreduce_sum_residual_gb300 as arn\n"
            f"arn.LIB_PATH = {str(tmp_path / 'missing.so')!r}\n"
            "try:\n    arn.ar_select_mode(8, 1, 7168)\nexcept RuntimeError as e:\n"
            "    print('raised:', 'not built' in str(e))\nelse:\n    print('no error')\n")
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.stdout.strip() == "raised: True", r.stdout + r.stderr


def test_the_environment_selects_the_checking_build():
    """ARN_CHECK_BUILD=1 makes the binding load libarnorm_check.so (bounds
    checks compiled in), so any program or test can run against it."""
    import subprocess
    import sys
    from allreduce_sum_residual_gb300 import _build
    _build.build(check=True)
    code = "import allreduce_sum_residual_gb300 as a; print(a.lib().ar_checks_bounds())"
    for flag, want in (("1", "1"), ("0", "0")):
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                           timeout=300, env={**os.environ, "ARN_CHECK_BUILD": flag})
        assert r.stdout.strip() == want, r.stdout + r.stderr
