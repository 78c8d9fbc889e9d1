"""Host-side checks of the CUDA library (no GPU needed).

The shared library must build for sm_103a, load, and export every function
include/attn_fwd.h declares; its host-only helpers (plan, work-item decoding,
argument checks that fail before any CUDA call) are checked here against the
work-decomposition numbers printed in "B200 Attention Kernel from Scratch to
Near-SOTA in 60 Diagrams", Chapter 14 (tests/golden/work_decomposition.txt).
"""
import ctypes
import math
import os
import re

import pytest

from dense_attention_forward_attn_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fwd.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "work_decomposition.txt")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(attn_[a-z_]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert "attn_fwd" in names and "attn_status_string" in names
    assert set(names) == set(attn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(attn.lib_path())
    for name in _declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert attn.status_string(code)
    assert attn.status_string(12345) == "unknown status"


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([c.strip() for c in line.split("|")])
    return rows


def test_plan_matches_worked_work_decomposition(lib):
    for name, B, H, S, value, _what in _golden_rows():
        B, H, S = int(B), int(H), int(S)
        p = attn.plan(B, H, S, S, 128, num_sms=148)
        if name.startswith("items_per_head"):
            assert p["work_items"] // (B * H) == int(value), name
        elif name.startswith("items_total"):
            assert p["work_items"] == int(value), name
        elif name.startswith("waves"):
            assert math.ceil(p["work_items"] / p["grid"]) == int(value), name
        elif name.startswith("kv_iters"):
            assert p["kv_tiles"] == int(value), name
        elif name.startswith("cta0_tiles"):
            tiles = []
            for item in range(0, 3 * p["grid"], p["grid"]):   # work_id += gridDim.x
                bh, qt0, n0, n1 = attn.work_item(item, B, H, S)
                tiles += [bh * p["q_tiles"] + qt0 + i for i in range(1 + (n1 > 0))]
            assert tiles == [int(t) for t in value.split(",")], name
        else:
            raise AssertionError(f"unknown golden row {name}")


def test_plan_resources_fit_one_sm(lib):
    p = attn.plan(4, 16, 4096, 4096, 128, num_sms=152)
    assert p["grid"] == 152 and p["work_items"] == 1024 and p["threads"] == 512
    assert p["smem_bytes"] <= 227 * 1024      # opt-in shared memory per block
    assert p["tmem_cols"] == 512              # S0 | S1 | O0 | O1, 128 columns each
    small = attn.plan(1, 2, 256, 256, 128, num_sms=152)
    assert small["grid"] == 2 and small["work_items"] == 2


def test_plan_ragged_lengths_round_tiles_up(lib):
    p = attn.plan(2, 3, 385, 129, 128, num_sms=152)
    assert p["q_tiles"] == 4 and p["kv_tiles"] == 2 and p["work_items"] == 2 * 3 * 2
    p = attn.plan(1, 1, 1, 1, 128, num_sms=152)
    assert p["q_tiles"] == 1 and p["kv_tiles"] == 1 and p["work_items"] == 1


def test_work_items_cover_every_q_tile_once(lib):
    for B, H, S in ((1, 3, 384), (2, 2, 1024), (1, 1, 128), (2, 1, 300), (1, 2, 1)):
        p = attn.plan(B, H, S, 128, 128, num_sms=152)
        assert p["kv_tiles"] == 1
        seen = set()
        for item in range(p["work_items"]):
            bh, qt0, n0, n1 = attn.work_item(item, B, H, S, 128)
            assert n0 == 1 and n1 in (0, 1)       # Sk = 128: one KV tile each
            for t in range(qt0, qt0 + 1 + (n1 > 0)):
                assert (bh, t) not in seen
                seen.add((bh, t))
        assert seen == {(bh, t) for bh in range(B * H) for t in range(-(-S // 128))}
        with pytest.raises(attn.AttnError):
            attn.work_item(p["work_items"], B, H, S, 128)


def _call(lib, q=16, k=32, v=48, o=64, lse=None, B=1, H=1, Sq=128, Sk=128, D=128, scale=0.1):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(q) if q else None, vp(k) if k else None, vp(v) if v else None,
                        vp(o) if o else None, vp(lse) if lse else None, B, H, Sq, Sk, D, scale, None)


def test_argument_checks_before_any_cuda_call(lib):
    big = 1 << 40   # fake, never dereferenced: every case below fails on the host first
    base = dict(q=big, k=2 * big, v=3 * big, o=4 * big)
    assert _call(lib, **base, D=64) == attn.ATTN_ERR_UNSUPPORTED
    assert _call(lib, **base, D=0) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **base, B=-1) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **base, Sk=0) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **base, scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **base, scale=float("inf")) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **base, scale=-0.5) == attn.ATTN_ERR_UNSUPPORTED
    assert _call(lib, **dict(base, q=0)) == attn.ATTN_ERR_INVALID_ARG
    assert _call(lib, **dict(base, o=big + 8)) == attn.ATTN_ERR_INVALID_ARG        # misaligned
    assert _call(lib, **dict(base, o=big + 4096)) == attn.ATTN_ERR_INVALID_ARG     # o overlaps q
    assert _call(lib, **base, lse=5 * big + 2) == attn.ATTN_ERR_INVALID_ARG        # misaligned lse
    assert _call(lib, **base, lse=4 * big + 64) == attn.ATTN_ERR_INVALID_ARG       # lse inside o


def test_flags_are_checked(lib):
    big = 1 << 40
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_ex(vp(big), vp(2 * big), vp(3 * big), vp(4 * big), None, 1, 1, 128, 128,
                         128, 0.1, 8, None)   # bit 3 is not a flag
    assert rc == attn.ATTN_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        attn._flags(False, "sbhd")
    assert attn._flags(True, "bshd") == attn.ATTN_FLAG_CAUSAL | attn.ATTN_FLAG_BSHD
    assert attn._flags(False, "bhsd", soft_exp2=True) == attn.ATTN_FLAG_SOFT_EXP2


def test_empty_problems_are_ok_without_launch(lib):
    assert _call(lib, q=0, k=0, v=0, o=0, B=0) == attn.ATTN_OK
    assert _call(lib, q=0, k=0, v=0, o=0, H=0) == attn.ATTN_OK
    assert _call(lib, q=0, k=0, v=0, o=0, Sq=0) == attn.ATTN_OK
    assert attn.plan(0, 4, 256, 256, 128, num_sms=152)["work_items"] == 0


def test_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 1, 128, 128, dtype=torch.float32)
    with pytest.raises(TypeError):
        attn.fwd(q, q, q)
    qb = torch.zeros(1, 1, 128, 256, dtype=torch.bfloat16)[..., :128]
    with pytest.raises(ValueError):
        attn.fwd(qb, qb, qb)


def test_causal_work_items_and_kv_tile_counts(lib):
    # top-left causal: Q tile t attends KV tiles 0..t (capped by the key count)
    for B, H, Sq, Sk in ((1, 2, 1024, 1024), (2, 1, 640, 300), (1, 1, 300, 900)):
        p = attn.plan(B, H, Sq, Sk, 128, num_sms=152, causal=True)
        kv = -(-Sk // 128)
        seen = {}
        for item in range(p["work_items"]):
            bh, qt0, n0, n1 = attn.work_item(item, B, H, Sq, Sk, causal=True)
            seen[(bh, qt0)] = (n0, n1)
            assert n0 == min(qt0 + 1, kv)
            assert n1 == (min(qt0 + 2, kv) if qt0 + 1 < p["q_tiles"] else 0)
        assert set(seen) == {(bh, 2 * i) for bh in range(B * H) for i in range(-(-p["q_tiles"] // 2))}
        # pairs numbered from the last one down: heaviest first when Sq == Sk (even tile count)
        work = [sum(attn.work_item(k, B, H, Sq, Sk, causal=True)[2:]) for k in range(p["work_items"])]
        if Sq == Sk:
            assert all(a >= b for a, b in zip(work, work[1:]))


def test_schedule_covers_every_item_once(lib):
    for items, grid in ((1024, 152), (1152, 152), (7, 152), (300, 16)):
        for causal in (False, True):
            got = []
            for cta in range(grid):
                r = 0
                while True:
                    k = attn.schedule(cta, r, grid, items, causal)
                    if k < 0:
                        break
                    got.append(k)
                    r += 1
            assert sorted(got) == list(range(items))
    # dense: static stride; causal: every other round reversed
    assert [attn.schedule(0, r, 148, 2048) for r in range(3)] == [0, 148, 296]
    assert [attn.schedule(0, r, 148, 2048, causal=True) for r in range(3)] == [0, 295, 296]


def _segments(cta, grid, items, n):
    out, r = [], 0
    while True:
        s = attn.segment(cta, r, grid, items, n)
        if s is None:
            return out
        out.append(s)
        r += 1


@pytest.mark.parametrize("items,grid,n", [
    (1024, 152, 32), (1024, 152, 64), (1024, 152, 128),   # S=4K/8K/16K at 16 heads
    (1152, 152, 96),                                     # S=12K, 24 heads: 7.58 rounds
    (1216, 152, 8),                                      # whole rounds: no split
    (400, 152, 3), (160, 152, 8), (301, 150, 5), (153, 152, 2), (1000, 7, 11),
])
def test_split_schedule_covers_every_unit_once_and_pairs_the_parts(lib, items, grid, n):
    """attn_fwd_ws's schedule: every (item, KV tile) unit runs exactly once; an item cut by KV range
    has exactly two parts, part 0 (from KV tile 0) ending the range of CTA `slot` and part 1
    (through the last KV tile) starting the range of CTA `slot + 1`; no CTA runs more units than
    the longest range of an even division of the last two rounds."""
    units = {}
    parts = {}
    per_cta = []
    for cta in range(grid):
        segs = _segments(cta, grid, items, n)
        total = 0
        for k, (item, j0, cnt, slot, part) in enumerate(segs):
            assert 0 <= item < items
            if cnt == -1:
                j0, cnt = 0, n
            assert 0 <= j0 and j0 + cnt <= n and cnt >= 1
            for j in range(j0, j0 + cnt):
                assert (item, j) not in units, (item, j)
                units[(item, j)] = cta
            total += cnt
            if cnt < n:
                assert slot >= 0 and part == (1 if j0 > 0 else 0)
                assert slot == (cta - 1 if part else cta) and 0 <= slot <= grid - 2
                if part == 1:
                    assert k == 0 or attn.segment(cta, k - 1, grid, items, n)[2] == -1  # first of the split rounds
                else:
                    assert k == len(segs) - 1 and j0 == 0
                assert (slot, part) not in parts
                parts[(slot, part)] = (item, j0, cnt)
            else:
                assert slot == -1
        per_cta.append(total)
    assert len(units) == items * n
    for (slot, part), (item, j0, cnt) in parts.items():
        other = parts[(slot, 1 - part)]
        assert other[0] == item
        lo, hi = (j0, j0 + cnt) if part == 0 else (other[1], other[1] + other[2])
        assert lo == 0 and hi == (other[1] if part == 0 else j0)
    full_rounds = -(-items // grid)
    if items > grid and items % grid and parts:
        sk0 = (items // grid - 1) * grid
        longest = (sk0 // grid) * n + -(-(items - sk0) * n // grid)
        assert max(per_cta) <= longest < full_rounds * n
    else:
        assert max(per_cta) == full_rounds * n


def test_split_schedule_is_used_where_it_pays(lib):
    # S=4K, S=8K and S=16K at 16 heads and S=12K at 24 heads split (the longest CTA gets >= 8
    # KV tiles shorter: 8, 16, 33 and 40); S=2K at 16 heads (4 tiles), whole rounds, short KV
    # ranges and causal calls do not
    def split(items, grid, n, causal=False):
        for c in range(grid):
            r = 0
            while (s := attn.segment(c, r, grid, items, n, causal)) is not None:
                if s[3] >= 0:
                    return True
                r += 1
        return False

    assert split(1024, 152, 128) and split(1024, 152, 64) and split(1024, 152, 32)
    assert not split(1024, 152, 16)
    assert split(1152, 152, 96)   # S=12K at 24 heads: 7.58 rounds
    assert not split(1216, 152, 96) and not split(400, 152, 1) and not split(100, 152, 8)
    assert not split(1024, 152, 128, causal=True)
    # 1136 items: 7.47 rounds, but 128 KV tiles per item gain 68 tiles from an even division
    assert split(1136, 152, 128)
    # 1144 items: 7.53 rounds of 32 tiles gain 15; 1100 items of 8 tiles gain 6, of 12 tiles 9
    assert split(1144, 152, 32)
    assert not split(1100, 152, 8) and split(1100, 152, 12)


def test_split_entry_point_checks_before_any_cuda_call(lib):
    big = 1 << 40
    vp = ctypes.c_void_p
    args = (vp(big), vp(2 * big), vp(3 * big), vp(4 * big), None, 1, 1, 128, 128, 64, 0.1, 0)
    assert lib.attn_fwd_ws(*args, None, 0, None) == attn.ATTN_ERR_UNSUPPORTED     # D = 64
    args = (vp(big), vp(2 * big), vp(3 * big), vp(4 * big), None, 1, 1, 128, 128, 128, 0.1, 8)
    assert lib.attn_fwd_ws(*args, None, 0, None) == attn.ATTN_ERR_INVALID_ARG     # bad flag
    n = ctypes.c_size_t(7)
    assert lib.attn_fwd_workspace(1, 1, 128, 128, 64, 0, ctypes.byref(n)) == attn.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_workspace(0, 1, 128, 128, 128, 0, ctypes.byref(n)) == attn.ATTN_OK and n.value == 0
    assert lib.attn_fwd_workspace(1, 1, 128, 128, 128, 0, None) == attn.ATTN_ERR_INVALID_ARG
    out = [ctypes.c_int() for _ in range(5)]
    assert lib.attn_fwd_segment(5, 0, 4, 10, 2, 0, *(ctypes.byref(x) for x in out)) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_segment(0, 0, 4, 10, 0, 0, *(ctypes.byref(x) for x in out)) == attn.ATTN_ERR_INVALID_ARG


# ------------------------------------------------------------- host-buffer forward planning

@pytest.mark.parametrize("B,H,S,expect", [
    (4, 16, 4096, (19, 4)),    # 16 items per head: 19 heads = 2 full rounds of 152
    (2, 16, 8192, (14, 3)),    # 32 per head: 14 heads = 448 items, 3 rounds
    (1, 16, 16384, (7, 3)),    # 64 per head: 7 heads = 448 items
])
def test_host_chunking_headline_shapes(lib, B, H, S, expect):
    per, n = attn.host_chunking(B, H, S, S, 152)
    assert (per, n) == expect
    # the chunked launches need no more grid rounds than one launch over everything
    units, per_unit = B * H, S // 256
    rounds = sum(-(-(min(per, units - u) * per_unit) // 152) for u in range(0, units, per))
    assert rounds == -(-(units * per_unit) // 152)


@pytest.mark.parametrize("B,H,Sq,Sk,layout,causal", [
    (1, 1, 128, 128, "bhsd", False), (3, 7, 300, 500, "bhsd", True), (2, 40, 1024, 1024, "bhsd", False),
    (4, 16, 4096, 4096, "bshd", False), (1, 200, 256, 128, "bhsd", False), (9, 3, 640, 640, "bshd", True),
])
def test_host_chunking_properties(lib, B, H, Sq, Sk, layout, causal):
    per, n = attn.host_chunking(B, H, Sq, Sk, 152, causal=causal, layout=layout)
    units = B if layout == "bshd" else B * H
    assert 1 <= n <= 8 and 1 <= per <= units
    assert per * n >= units and per * (n - 1) < units


def test_host_workspace_bytes(lib):
    ws = ctypes.c_size_t()
    assert lib.attn_fwd_host_workspace(2, 3, 300, 500, 128, 0, ctypes.byref(ws)) == attn.ATTN_OK
    al = lambda x: (x + 255) // 256 * 256
    q, kv, l = 6 * 300 * 128 * 2, 6 * 500 * 128 * 2, 6 * 300 * 4
    assert ws.value == al(q) + 2 * al(kv) + al(q) + al(l)
    assert lib.attn_fwd_host_workspace(2, 3, 300, 500, 64, 0, ctypes.byref(ws)) == attn.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_host_workspace(2, 3, 300, 500, 128, 8, ctypes.byref(ws)) == attn.ATTN_ERR_INVALID_ARG


def test_host_batch_order_puts_most_work_per_byte_first():
    """fwd_host_batch's default enqueue order: problems with more tensor work per copied byte
    first, so their kernels run while the other problems' copies stream in; a bad explicit
    order is rejected before any CUDA call."""
    import torch
    def pb(B, H, Sq, Sk, causal=False, layout="bhsd"):
        qs = (B, Sq, H, 128) if layout == "bshd" else (B, H, Sq, 128)
        ks = (B, Sk, H, 128) if layout == "bshd" else (B, H, Sk, 128)
        z = lambda sh: torch.empty(sh, dtype=torch.bfloat16)
        return dict(q=z(qs), k=z(ks), v=z(ks), causal=causal, layout=layout)
    probs = [pb(4, 16, 64, 64), pb(1, 16, 256, 256), pb(2, 16, 128, 128)]
    assert attn.batch_order(probs) == [1, 2, 0]
    # the causal mask halves the work: S=256 causal ranks with S=128 dense (stable order)
    probs = [pb(1, 2, 128, 128), pb(1, 2, 256, 256, causal=True), pb(1, 2, 64, 64, layout="bshd")]
    assert attn.batch_order(probs) == [0, 1, 2]
    with pytest.raises(ValueError):
        attn.fwd_host_batch(probs, order=[0, 0, 1])


def test_bench_source_hash_ignores_comments(tmp_path, monkeypatch):
    """The hash that decides whether the recorded DRAM traffic still describes the kernel changes
    with the kernel's code, not with its comments or blank lines."""
    import shutil
    import bench
    csrc = tmp_path / "dense_attention_forward_attn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(ROOT, "dense_attention_forward_attn_gb300", "csrc")
    for name in ("attn_fwd_kernel.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(src, name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench._source_sha()
    k = csrc / "attn_fwd_kernel.cuh"
    text = k.read_text()
    k.write_text("// a new comment\n\n" + text.replace("namespace attn {", "namespace attn {  /* note */", 1))
    assert bench._source_sha() == base
    k.write_text(text.replace("kRebaseThresholdLog2 = 8.0f", "kRebaseThresholdLog2 = 7.0f", 1))
    assert bench._source_sha() != base


def test_workspace_query_needs_no_launch(lib):
    # empty problems need no workspace; a bad head size is refused before any CUDA call
    assert attn.workspace_bytes(0, 16, 4096, 4096) == 0
    with pytest.raises(attn.AttnError):
        attn.workspace_bytes(1, 1, 128, 128, D=64)


def test_bench_config_names_each_rows_mask_and_layout():
    # the JSON line's per-shape config states the row's causal flag and tensor layout
    import bench
    from dense_attention_forward_attn_gb300 import workloads as wl
    dense = bench.bench_config("w", wl.HEADLINE, 24, 1)
    assert [d["causal"] for d in dense["shapes"]] == [False] * len(wl.HEADLINE)
    assert {d["layout"] for d in dense["shapes"]} == {"BHSD contiguous"}
    causal = bench.bench_config("w", wl.HEADLINE, 24, 1, causal=True, layout="bshd")
    assert all(d["causal"] for d in causal["shapes"])
    assert {d["layout"] for d in causal["shapes"]} == {"BSHD contiguous"}
    assert causal["parallelism"] == "single GPU" and dense["problems_per_shape_per_step"] == 24
