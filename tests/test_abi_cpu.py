"""The C-ABI library loads, exports every declared symbol, and its host-side
logic (argument checks, status codes, launch-geometry planning) behaves --
all without a GPU.  No call here launches a kernel: every call either fails
validation before any CUDA call or is a plan query with an explicit SM count.
"""
import ctypes
import os
import re

import pytest

import gated_activation_gb300 as ga
from gated_activation_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gated_act.h")
TEST_HEADER = os.path.join(ROOT, "include", "gated_act_testing.h")
GB300_SMS = 152


@pytest.fixture(scope="module")
def lib():
    if not gbuild.up_to_date():
        gbuild.build()
    return ga.load_library()


def declared_functions(headers=None) -> list[str]:
    """Functions declared in the given headers (default: every include/*.h)."""
    if headers is None:
        inc = os.path.join(ROOT, "include")
        headers = [os.path.join(inc, f) for f in sorted(os.listdir(inc)) if f.endswith(".h")]
    names = set()
    for h in headers:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_test_hooks_stay_out_of_the_product_header():
    product = declared_functions([HEADER])
    hooks = declared_functions([TEST_HEADER])
    assert hooks and all("selftest" in n for n in hooks)
    assert not [n for n in product if "selftest" in n]


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ("gelu_and_mul_sparse", "silu_and_mul", "gated_act_status_string",
                 "gelu_and_mul_sparse_ex", "gelu_and_mul_sparse_plan",
                 "gated_act_last_cuda_error"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(declared_functions()) == set(ga.EXPORTED)


def test_status_codes_match_the_header():
    """Every GATED_ACT_ status the header declares has the same value in the binding."""
    with open(HEADER) as f:
        text = f.read()
    body = text[text.index("typedef enum gated_act_status"):text.index("} gated_act_status;")]
    codes = dict(re.findall(r"GATED_ACT_(\w+)\s*=\s*(-?\d+)", body))
    assert len(codes) >= 13, codes
    for name, value in codes.items():
        assert getattr(ga, name) == int(value), name


def test_status_strings(lib):
    for code in range(-12, 1):
        s = lib.gated_act_status_string(code)
        assert s and s.decode()
    assert lib.gated_act_status_string(-99).decode() == "unknown status"
    assert lib.gated_act_last_cuda_error() == 0


def _gelu(lib, out, inp, T, d, rs, z=1.0):
    return lib.gelu_and_mul_sparse(out, inp, T, d, rs, z, None)


@pytest.mark.parametrize("T,d,rs,code", [
    (-1, 8, 16, ga.ERR_SIZE), (4, 0, 16, ga.ERR_SIZE), (4, -3, 16, ga.ERR_SIZE),
    (4, 8, 15, ga.ERR_STRIDE), (4, 8, 0, ga.ERR_STRIDE),
    (4, (1 << 30) + 8, 1 << 32, ga.ERR_TOO_LARGE),
])
def test_gelu_rejects_bad_sizes(lib, T, d, rs, code):
    assert _gelu(lib, 0x1000, 0x100000, T, d, rs) == code


def test_gelu_rejects_null_odd_and_overlapping_pointers(lib):
    assert _gelu(lib, None, 0x100000, 4, 8, 16) == ga.ERR_NULL
    assert _gelu(lib, 0x1000, None, 4, 8, 16) == ga.ERR_NULL
    assert _gelu(lib, 0x1001, 0x100000, 4, 8, 16) == ga.ERR_ALIGN
    assert _gelu(lib, 0x1000, 0x100001, 4, 8, 16) == ga.ERR_ALIGN
    # in spans [0x10000, 0x10000 + 2*(3*16+16)) = 128 B; out [.., +64 B)
    assert _gelu(lib, 0x10000 + 64, 0x10000, 4, 8, 16) == ga.ERR_OVERLAP
    assert _gelu(lib, 0x10000 - 63, 0x10000, 4, 8, 16) == ga.ERR_ALIGN
    assert _gelu(lib, 0x10000 - 62, 0x10000, 4, 8, 16) == ga.ERR_OVERLAP


def test_zero_rows_is_a_no_op(lib):
    assert _gelu(lib, None, None, 0, 8, 16) == ga.OK
    assert lib.silu_and_mul(None, None, 0, 8, None) == ga.OK


@pytest.mark.parametrize("M,d,code", [(-1, 8, ga.ERR_SIZE), (4, 0, ga.ERR_SIZE),
                                      (4, (1 << 30) + 1, ga.ERR_TOO_LARGE)])
def test_silu_rejects_bad_sizes(lib, M, d, code):
    assert lib.silu_and_mul(0x1000, 0x100000, M, d, None) == code


def test_silu_rejects_null_odd_and_overlap(lib):
    assert lib.silu_and_mul(None, 0x100000, 4, 8, None) == ga.ERR_NULL
    assert lib.silu_and_mul(0x1001, 0x100000, 4, 8, None) == ga.ERR_ALIGN
    assert lib.silu_and_mul(0x100000 + 100, 0x100000, 4, 8, None) == ga.ERR_OVERLAP


def test_widened_rows_reject_bad_arguments(lib):
    # silu_and_mul_bounded needs a live-count pointer, aligned to 4
    assert lib.silu_and_mul_bounded(0x1000, 0x100000, 4, 8, None, None) == ga.ERR_NULL
    assert lib.silu_and_mul_bounded(0x1000, 0x100000, 4, 8, 0x2002, None) == ga.ERR_ALIGN
    assert lib.silu_and_mul_bounded(0x1000, 0x100000, -1, 8, 0x2000, None) == ga.ERR_SIZE
    assert lib.silu_and_mul_bounded(None, None, 0, 8, None, None) == ga.OK
    # gelu_and_mul takes a row stride
    assert lib.gelu_and_mul(0x1000, 0x100000, 4, 8, 15, None) == ga.ERR_STRIDE
    assert lib.gelu_and_mul(0x1000, 0x100000, 4, 0, 16, None) == ga.ERR_SIZE
    assert lib.gelu_and_mul(0x100000 + 8, 0x100000, 4, 8, 16, None) == ga.ERR_OVERLAP
    assert lib.gelu_and_mul(None, None, 0, 8, 16, None) == ga.OK
    # squared_relu is not gated: [M, d] -> [M, d]
    assert lib.squared_relu(0x1000, 0x100000, 4, 0, None) == ga.ERR_SIZE
    assert lib.squared_relu(None, 0x100000, 4, 8, None) == ga.ERR_NULL
    assert lib.squared_relu(0x100000 + 62, 0x100000, 4, 8, None) == ga.ERR_OVERLAP


def plan(lib, T, d, rs=None, variant=0, cluster=0, sms=GB300_SMS, out=0x10000, inp=0x100000,
         dtype=0, ws=0):
    p = ga.Plan()
    if ws:
        rc = lib.gelu_and_mul_sparse_plan_ex(out, inp, T, d, rs or 2 * d, dtype, variant, cluster,
                                             sms, 1, ctypes.byref(p))
    else:
        rc = lib.gelu_and_mul_sparse_plan(out, inp, T, d, rs or 2 * d, dtype, variant, cluster,
                                          sms, ctypes.byref(p))
    return rc, p.as_dict()


def test_plan_geometry_families(lib):
    # short rows: a warp per row
    rc, p = plan(lib, 2048, 512)
    assert rc == 0 and p["variant"] == "warp_rows" and p["vec_per_thread"] == 2
    # d = 2048 .. 8192 at any T: one CTA per row, one row per CTA
    for T, d in ((2048, 2048), (2048, 8192), (64, 8192), (1, 4096)):
        rc, p = plan(lib, T, d)
        assert rc == 0 and p["variant"] == "cta_row" and p["cluster"] == 1 and p["grid"] == T
    # the widest rows at many rows per SM (no workspace): persistent TMA rows,
    # one wave of CTAs
    rc, p = plan(lib, 2048, 32768)
    assert rc == 0 and p["variant"] == "tma_rows" and p["threads"] == 1024
    assert p["grid"] == GB300_SMS and p["stages"] >= 2 and p["smem_bytes"] <= 227 * 1024
    # d = 14336 .. 16384 from 8 rows per SM on: producer/consumer rows, one CTA
    # per SM of 16 consumer warps, a ring of four slots
    rc, p = plan(lib, 2048, 16384)
    assert rc == 0 and p["variant"] == "pipe_rows" and p["threads"] == 544
    assert p["ctas_per_sm"] == 1 and p["stages"] == 4 and p["grid"] == GB300_SMS
    # rows wider than 16384 at fewer rows per SM: the producer/consumer rows
    rc, p = plan(lib, 512, 32768)
    assert rc == 0 and p["variant"] == "pipe_rows" and p["threads"] == 544
    rc, p = plan(lib, 1024, 16384)
    assert rc == 0 and p["variant"] == "cta_row" and p["threads"] == 512
    # a handful of wide rows: 8-CTA clusters per row
    rc, p = plan(lib, 1, 32768)
    assert rc == 0 and p["variant"] == "cta_row" and p["cluster"] == 8
    # 9 to 32 rows of d >= 32768: split rows of 8 (to 19 rows) or 4 CTAs
    for T, c in ((9, 8), (19, 8), (20, 4), (32, 4)):
        rc, p = plan(lib, T, 32768)
        assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == c, T
    # 33 rows of d > 16384 and more, while two CTAs per row fit one wave:
    # split rows, two independent CTAs per row; beyond, one CTA per row
    for T in (33, 48, 64, 76):
        rc, p = plan(lib, T, 32768)
        assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == 2, T
        assert p["grid"] == 2 * T and p["threads"] == 512 and p["vec_per_thread"] == 8
    assert plan(lib, 77, 32768)[1]["variant"] == "cta_row"
    assert plan(lib, 77, 32768)[1]["cluster"] == 1
    # d = 16384: split rows with the most CTAs per row (8, 4, 2) that fit one
    # wave of the SMs
    for T, c in ((1, 8), (8, 8), (9, 8), (19, 8), (20, 4), (38, 4), (39, 2), (64, 2), (76, 2)):
        rc, p = plan(lib, T, 16384)
        assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == c, (T, p)
        assert p["threads"] == 256 and p["grid"] == c * T
    assert plan(lib, 77, 16384)[1]["variant"] == "cta_row"
    # rows wider than one CTA's registers are split across a cluster
    rc, p = plan(lib, 2048, 65536, variant=ga.VARIANT_CTA_ROW)
    assert rc == 0 and p["cluster"] == 2 and p["grid"] == 4096


def test_plan_covers_every_slice(lib):
    # threads x vectors of each CTA slice cover the row for every aligned d
    for d in list(range(8, 4096, 8)) + [8192, 8200, 16384, 16392, 32768, 65536, 131072, 262144]:
        for T in (1, 8, 64, 2048):
            rc, p = plan(lib, T, d)
            assert rc == 0
            nvec = d // 8
            if p["variant"] == "warp_rows":
                assert 32 * p["vec_per_thread"] >= nvec
            elif p["variant"] == "tma_rows":
                assert p["threads"] * p["vec_per_thread"] >= nvec and p["vec_per_thread"] <= 4
                # every CTA of an SM fits: slots of 2d bytes plus their barriers
                assert p["smem_bytes"] == p["stages"] * (2 * d + 8)
                assert p["stages"] >= 2 and p["smem_bytes"] <= 227 * 1024 - 1024
            elif p["variant"] == "pipe_rows":
                # consumer threads (all warps but the producer's) cover the row
                assert (p["threads"] - 32) * p["vec_per_thread"] >= nvec
                assert p["smem_bytes"] == p["stages"] * (2 * d + 24) and p["stages"] >= 3
            elif p["variant"] == "cta_row":
                sv = -(-nvec // p["cluster"])
                assert p["threads"] * p["vec_per_thread"] >= sv
                assert p["threads"] <= 1024 and p["cluster"] <= 8
                assert p["grid"] % p["cluster"] == 0
            elif p["variant"] == "split_rows":
                # every CTA holds the whole row's gate for the statistics
                assert p["threads"] * p["vec_per_thread"] >= nvec
                assert p["cluster"] in (2, 4, 8) and p["grid"] == T * p["cluster"]
            else:
                pytest.fail(f"aligned d={d} fell back to scalar")


def test_plan_eight_cta_clusters_use_two_vector_slices(lib):
    # a handful of 32768-wide rows: 8-CTA clusters of 256 threads holding two
    # 16-byte vectors each (512-vector slices)
    for T in (1, 8):
        rc, p = plan(lib, T, 32768)
        assert rc == 0 and p["cluster"] == 8 and p["threads"] == 256 and p["vec_per_thread"] == 2
    # 4-CTA clusters (forced) keep four vectors per thread
    rc, p = plan(lib, 16, 32768, variant=ga.VARIANT_CTA_ROW, cluster=4)
    assert rc == 0 and p["cluster"] == 4 and p["vec_per_thread"] == 4
    # up to 8 rows of 24576 and more: 8-CTA clusters of two-vector threads
    for T in (1, 8):
        rc, p = plan(lib, T, 24576)
        assert rc == 0 and p["variant"] == "cta_row" and p["cluster"] == 8, (T, p)
    # above 8192 up to 16384: 8-CTA clusters up to 8 rows, 16 rows, and 32
    # rows from 14336
    rc, p = plan(lib, 8, 4096)
    assert rc == 0 and p["variant"] == "cta_row" and p["cluster"] == 1
    # from d = 8192: split rows, the most CTAs per row that fit one wave; at
    # d = 8192 only 8 or 4 of them
    for T, d, c in ((1, 9216, 8), (8, 14336, 8), (9, 9216, 8), (16, 11008, 8), (17, 11008, 8),
                    (24, 12288, 4), (38, 14336, 4), (39, 14336, 2), (76, 9216, 2), (9, 8192, 8),
                    (38, 8192, 4), (1, 20480, 8), (8, 20480, 8), (1, 8192, 8), (8, 8192, 8)):
        rc, p = plan(lib, T, d)
        assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == c, (T, d, p)
    for T, d in ((39, 8192), (77, 11008), (64, 4096)):
        assert plan(lib, T, d)[1]["variant"] == "cta_row", (T, d)
    # without a workspace, many rows of d >= 28672 take tma rows
    assert plan(lib, 2048, 28672)[1]["variant"] == "tma_rows"
    assert plan(lib, 1219, 28672)[1]["variant"] == "tma_rows"
    assert plan(lib, 1215, 28672)[1]["variant"] == "pipe_rows"
    assert plan(lib, 2048, 28672, ws=1)[1]["variant"] == "pipe_rows"
    # between 16384 and 32768: split rows of 8 CTAs to 19 rows, of 4 to 32,
    # of 2 while they fit one wave; then one CTA per row
    for d in (20480, 24576):
        for T, c in ((16, 8), (24, 4), (33, 2)):
            rc, p = plan(lib, T, d)
            assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == c, (T, d, p)
        assert plan(lib, 77, d)[1]["cluster"] == 1


def test_plan_split_rows_forced_and_refused(lib):
    # forced: any C of 2, 4, 8 for rows of up to 4096 vectors
    for d, c, nt in ((1024, 2, 256), (1024, 8, 128), (8192, 8, 128), (8192, 4, 256),
                     (16384, 4, 256), (16392, 8, 512), (32768, 2, 512)):
        rc, p = plan(lib, 5, d, variant=ga.VARIANT_SPLIT_ROWS, cluster=c)
        assert rc == 0 and p["variant"] == "split_rows" and p["cluster"] == c, (d, p)
        assert p["threads"] == nt and p["grid"] == 5 * c
    for d, c in ((16384, 0), (16384, 3), (16384, 16), (32776, 2), (16384 + 4, 2)):
        assert plan(lib, 5, d, variant=ga.VARIANT_SPLIT_ROWS, cluster=c)[0] == ga.ERR_VARIANT
    # native mode: split rows of 8 or 4 CTAs, one CTA per row where they
    # would take two at d <= 16384
    for T, want in ((16, (ga.VARIANT_SPLIT_ROWS, 8)), (32, (ga.VARIANT_SPLIT_ROWS, 4)),
                    (64, (ga.VARIANT_CTA_ROW, 1))):
        p = ga.Plan()
        assert lib.gelu_and_mul_sparse_native_plan(0x10000, 0x100000, T, 16384, 32768, ga.BF16,
                                                   GB300_SMS, ctypes.byref(p)) == ga.OK
        assert (p.variant, p.cluster) == want, (T, p.as_dict())
    # fp16 rows of the same width take split rows too; fp32 rows of 8192
    # (the same 2048 vectors) as well
    assert plan(lib, 16, 16384, dtype=ga.F16)[1]["variant"] == "split_rows"
    assert plan(lib, 16, 8192, dtype=ga.F32)[1]["variant"] == "split_rows"


def test_plan_falls_back_to_scalar(lib):
    assert plan(lib, 4, 31)[1]["variant"] == "scalar"            # d not a multiple of 8
    assert plan(lib, 4, 64, rs=130)[1]["variant"] == "scalar"    # row stride not 16-byte
    assert plan(lib, 4, 64, inp=0x100002)[1]["variant"] == "scalar"   # misaligned pointer
    assert plan(lib, 4, 262144 + 8)[1]["variant"] == "scalar"    # wider than 8 CTAs hold


def test_plan_tma_rows_limits(lib):
    for d in (64, 1024, 2048, 8192, 16384, 32768):
        rc, p = plan(lib, 4096, d, variant=ga.VARIANT_TMA_ROWS)
        assert rc == 0 and p["variant"] == "tma_rows"
        cps = -(-p["grid"] // GB300_SMS)
        assert cps * p["threads"] <= 2048 and cps * (p["smem_bytes"] + 1024) <= 228 * 1024
    assert plan(lib, 4096, 32776, variant=ga.VARIANT_TMA_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4096, 31, variant=ga.VARIANT_TMA_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4096, 64, rs=130, variant=ga.VARIANT_TMA_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 5, 8192, variant=ga.VARIANT_TMA_ROWS)[1]["grid"] == 5


def test_plan_typed(lib):
    # fp16 rows use the CTA-row geometry, fp32 rows hold 4 elements per vector
    rc, p = plan(lib, 2048, 16384, dtype=ga.F16)
    assert rc == 0 and p["variant"] == "cta_row" and p["threads"] == 512
    rc, p = plan(lib, 2048, 16384, dtype=ga.F32)
    assert rc == 0 and p["variant"] == "cta_row" and p["threads"] == 1024 and p["cluster"] == 1
    rc, p = plan(lib, 2048, 32768, dtype=ga.F32)
    assert rc == 0 and p["cluster"] == 2
    assert plan(lib, 4, 6, dtype=ga.F32)[1]["variant"] == "scalar"      # d not a multiple of 4
    assert plan(lib, 4, 12, dtype=ga.F32)[1]["variant"] == "cta_row"
    assert plan(lib, 4, 64, dtype=ga.F16, variant=ga.VARIANT_TMA_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, dtype=ga.F32, variant=ga.VARIANT_WARP_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, dtype=3)[0] == ga.ERR_DTYPE
    # typed validation: fp32 pointers must be 4-byte aligned
    assert lib.gelu_and_mul_sparse_typed(0x1002, 0x100000, 4, 8, 16, 1.0, ga.F32, 0, 0,
                                         None) == ga.ERR_ALIGN
    assert lib.gelu_and_mul_sparse_typed(0x100000 + 120, 0x100000, 4, 8, 16, 1.0, ga.F32, 0, 0,
                                         None) == ga.ERR_OVERLAP


def test_native_rounding_rejects_fp32_and_bad_args(lib):
    assert lib.gelu_and_mul_sparse_native(0x1000, 0x100000, 4, 8, 16, 1.0, ga.F32,
                                          None) == ga.ERR_DTYPE
    assert lib.gelu_and_mul_sparse_native(0x1000, 0x100000, 4, 8, 15, 1.0, ga.BF16,
                                          None) == ga.ERR_STRIDE
    assert lib.gelu_and_mul_sparse_native(None, None, 0, 8, 16, 1.0, ga.F16, None) == ga.OK


def test_plan_forced_variants(lib):
    assert plan(lib, 4, 2048, variant=ga.VARIANT_CTA_ROW, cluster=2)[1]["cluster"] == 2
    assert plan(lib, 4, 4096, variant=ga.VARIANT_WARP_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, variant=ga.VARIANT_CTA_ROW, cluster=3)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, variant=ga.VARIANT_CTA_ROW, cluster=16)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 65536, variant=ga.VARIANT_CTA_ROW, cluster=1)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 31, variant=ga.VARIANT_WARP_ROWS)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, variant=9)[0] == ga.ERR_VARIANT
    assert plan(lib, 4, 64, variant=ga.VARIANT_SCALAR)[1]["variant"] == "scalar"


def test_plan_depends_only_on_arguments(lib):
    a = plan(lib, 64, 8192)
    b = plan(lib, 64, 8192)
    assert a == b
    # a different SM count may change the choice, never the validity
    rc, p = plan(lib, 2048, 32768, sms=32)
    assert rc == 0 and p["variant"] == "tma_rows" and p["grid"] == 32
    rc, p = plan(lib, 1024, 32768, sms=1024)
    assert rc == 0 and p["variant"] == "cta_row"


def test_workspace_entry_rejects_bad_workspaces(lib):
    assert lib.gelu_and_mul_sparse_workspace_bytes() == 16
    # no workspace, or one that is not 8-byte aligned: refused before any launch
    assert lib.gelu_and_mul_sparse_ws(0x1000, 0x100000, 4, 8, 16, 1.0, ga.BF16, 0, 0,
                                      None, None) == ga.ERR_NULL
    assert lib.gelu_and_mul_sparse_ws(0x1000, 0x100000, 0, 8, 16, 1.0, ga.BF16, 0, 0,
                                      0x2004, None) == ga.ERR_ALIGN
    # sizes are validated before the workspace
    assert lib.gelu_and_mul_sparse_ws(0x1000, 0x100000, -1, 8, 16, 1.0, ga.BF16, 0, 0,
                                      0x2000, None) == ga.ERR_SIZE


def test_plan_reports_dynamic_rows(lib):
    # d = 32768 bf16 on a 152-SM device without a workspace: TMA rows from 8
    # rows per SM on, so eight or more per CTA: rows would be taken
    # dynamically given a workspace (which picks pipe rows instead)
    for T in (1216, 2048, 4096):
        p = ga.Plan()
        assert lib.gelu_and_mul_sparse_plan_ex(0x1000, 0x10000000, T, 32768, 65536, ga.BF16,
                                               0, 0, 152, 0, ctypes.byref(p)) == ga.OK
        assert p.variant == ga.VARIANT_TMA_ROWS and p.grid == 152 and p.dynamic_rows == 1
    # forced TMA rows below six rows per CTA with a workspace: still dynamic
    p = ga.Plan()
    assert lib.gelu_and_mul_sparse_plan_ex(0x1000, 0x10000000, 400, 16384, 32768, ga.BF16,
                                           ga.VARIANT_TMA_ROWS, 0, 152, 1,
                                           ctypes.byref(p)) == ga.OK
    assert p.variant == ga.VARIANT_TMA_ROWS and p.dynamic_rows == 1
    # a forced bulk-copy geometry always takes rows dynamically; others never
    p = ga.Plan()
    assert lib.gelu_and_mul_sparse_plan(0x1000, 0x10000000, 10, 4096, 8192, ga.BF16,
                                        ga.VARIANT_TMA_ROWS, 0, 152, ctypes.byref(p)) == ga.OK
    assert p.dynamic_rows == 1
    assert lib.gelu_and_mul_sparse_plan(0x1000, 0x10000000, 10, 4096, 8192, ga.BF16,
                                        ga.VARIANT_CTA_ROW, 1, 152, ctypes.byref(p)) == ga.OK
    assert p.dynamic_rows == 0


def _plan_ex(lib, T, d, ws, variant=0, cluster=0):
    p = ga.Plan()
    rc = lib.gelu_and_mul_sparse_plan_ex(0x1000, 0x10000000, T, d, 2 * d, ga.BF16, variant,
                                         cluster, 152, ws, ctypes.byref(p))
    return rc, p


def test_plan_pipe_rows_choice(lib):
    # rows wider than 16384 from ~1.6 rows per SM (d = 32768) on: pipe rows,
    # one CTA per SM of 16 consumer warps + 1 producer warp, rows always
    # dynamic given a workspace
    for T, ws, want in ((200, 1, ga.VARIANT_CTA_ROW), (256, 1, ga.VARIANT_PIPE_ROWS),
                        (1024, 0, ga.VARIANT_PIPE_ROWS), (1024, 1, ga.VARIANT_PIPE_ROWS),
                        (2048, 1, ga.VARIANT_PIPE_ROWS), (2048, 0, ga.VARIANT_TMA_ROWS),
                        (4096, 0, ga.VARIANT_TMA_ROWS)):
        rc, p = _plan_ex(lib, T, 32768, ws)
        assert rc == ga.OK and p.variant == want, (T, ws, p.variant)
        if want == ga.VARIANT_PIPE_ROWS:
            assert (p.threads, p.vec_per_thread, p.ctas_per_sm, p.grid) == (544, 8, 1, 152)
            assert p.dynamic_rows == 1 and p.stages == 3
    # narrower than 32768 but wider than 16384: pipe rows with or without one
    for d in (20480, 24576):
        for ws in (0, 1):
            assert _plan_ex(lib, 2048, d, ws)[1].variant == ga.VARIANT_PIPE_ROWS
    # d = 14336 .. 16384: from 8 rows per SM on, with or without a
    # workspace; one CTA per SM, four slots
    for T, d, ws, want in ((1216, 16384, 1, True), (1215, 16384, 1, False),
                           (1216, 16384, 0, True), (1215, 16384, 0, False),
                           (2048, 12288, 1, False), (2048, 12288, 0, False),
                           (2048, 14336, 0, True), (4096, 10240, 1, False)):
        rc, p = _plan_ex(lib, T, d, ws)
        assert rc == ga.OK and (p.variant == ga.VARIANT_PIPE_ROWS) == want, (T, d, ws)
        if want:
            assert p.ctas_per_sm == 1 and p.stages == 4
    # d <= 8192 never picks pipe rows by itself
    for d in (2048, 4096, 8192):
        for ws in (0, 1):
            assert _plan_ex(lib, 4096, d, ws)[1].variant != ga.VARIANT_PIPE_ROWS


def test_plan_pipe_rows_limits(lib):
    # every forced setting fits the SM: threads, registers (launch bounds),
    # shared memory with its per-CTA reserve, three slots or more
    budget = {4: 4, 8: 2, 16: 1}
    for d in (64, 1000, 2048, 4096, 8192, 12296, 16384, 24576, 32768):
        for cps in (0, 1, 2, 4, 8):
            rc, p = _plan_ex(lib, 4096, d, 1, ga.VARIANT_PIPE_ROWS, cps)
            if rc != ga.OK:
                assert rc == ga.ERR_VARIANT
                continue
            ncw = p.threads // 32 - 1
            assert p.variant == ga.VARIANT_PIPE_ROWS and ncw in budget
            assert p.ctas_per_sm <= budget[ncw] and (cps == 0 or p.ctas_per_sm == cps)
            assert ncw * 32 * p.vec_per_thread >= d // 8
            assert p.stages >= 3 and p.ctas_per_sm * (p.smem_bytes + 1024 + 256) <= 228 * 1024
            assert p.smem_bytes == p.stages * (2 * d + 24)
        assert _plan_ex(lib, 4096, d, 1, ga.VARIANT_PIPE_ROWS, 0)[0] == ga.OK
    assert _plan_ex(lib, 4096, 32776, 1, ga.VARIANT_PIPE_ROWS)[0] == ga.ERR_VARIANT
    assert _plan_ex(lib, 4096, 32768, 1, ga.VARIANT_PIPE_ROWS, 2)[0] == ga.ERR_VARIANT
    assert _plan_ex(lib, 4096, 64, 1, ga.VARIANT_PIPE_ROWS, 3)[0] == ga.ERR_VARIANT
    assert _plan_ex(lib, 4096, 64, 1, ga.VARIANT_PIPE_ROWS, 16)[0] == ga.ERR_VARIANT
    p = ga.Plan()
    assert lib.gelu_and_mul_sparse_plan_ex(0x1000, 0x100000, 4, 64, 128, ga.F16,
                                           ga.VARIANT_PIPE_ROWS, 0, 152, 1,
                                           ctypes.byref(p)) == ga.ERR_VARIANT


def test_native_plan(lib):
    # native rows run one CTA (or cluster) per row at every width, where the
    # plain call streams the widest rows through the bulk-copy kernels (pipe
    # rows with the table-read epilogue were measured slower: 2048 x 16384
    # 41.3 against 34.6 us)
    p = ga.Plan()
    for T, d in ((2048, 16384), (1300, 14336), (1024, 32768), (2048, 32768), (4096, 64),
                 (1, 32768)):
        assert lib.gelu_and_mul_sparse_native_plan(0, 0x100000, T, d, 2 * d, ga.BF16,
                                                   GB300_SMS, ctypes.byref(p)) == 0
        assert ga.VARIANT_NAMES[p.variant] == "cta_row", (T, d)
    assert lib.gelu_and_mul_sparse_native_plan(0, 0x100000, 1, 32768, 65536, ga.BF16,
                                               GB300_SMS, ctypes.byref(p)) == 0
    assert p.cluster == 8
    assert lib.gelu_and_mul_sparse_native_plan(0, 0x100000, 2048, 16384, 32768, ga.F16,
                                               GB300_SMS, ctypes.byref(p)) == 0
    assert ga.VARIANT_NAMES[p.variant] == "cta_row"
    assert lib.gelu_and_mul_sparse_native_plan(0, 0x100000, 4, 64, 128, ga.F32, GB300_SMS,
                                               ctypes.byref(p)) == ga.ERR_DTYPE
    assert lib.gelu_and_mul_sparse_native_plan(0, 0x100000, 4, 64, 128, ga.BF16, GB300_SMS,
                                               None) == ga.ERR_NULL


def _native_plan(lib, T, d, dtype, sms=GB300_SMS):
    p = ga.Plan()
    rc = lib.gelu_and_mul_sparse_native_plan(0x10000, 0x100000, T, d, 2 * d, dtype, sms,
                                             ctypes.byref(p))
    return rc, p.as_dict()


@pytest.mark.parametrize("dtype", [ga.BF16, ga.F16, ga.F32])
def test_plan_invariants_over_modes(lib, dtype):
    """Every automatic plan -- each element type, plain and native rounding,
    with and without a workspace, across row counts around the SM count and
    its multiples -- is a launch the kernels can run: a legal block, a grid
    that covers the rows, CTA slices that cover the row, shared memory within
    the SM's limit, and only the geometries each mode has."""
    elem = 4 if dtype == ga.F32 else 2
    epv = 16 // elem
    Ts = (1, 2, 8, 9, 19, 33, 64, 76, 77, 152, 153, 456, 1216, 1217, 2048, 4096)
    ds = (64, 512, 1000, 2048, 4096, 6144, 8192, 9216, 11008, 14336, 16384, 20480, 24576,
          28672, 32768, 65536)
    modes = [("plain", 0), ("plain", 1)] + ([("native", 0)] if dtype != ga.F32 else [])
    for mode, ws in modes:
        for T in Ts:
            for d in ds:
                if mode == "native":
                    rc, p = _native_plan(lib, T, d, dtype)
                else:
                    rc, p = plan(lib, T, d, dtype=dtype, ws=ws)
                where = (mode, ws, T, d, p)
                assert rc == 0, where
                v, nt, grid = p["variant"], p["threads"], p["grid"]
                assert 32 <= nt <= 1024 and nt % 32 == 0, where
                assert 1 <= grid <= 0x7FFFFFFF, where
                nvec = d // epv
                if d % epv:
                    assert v == "scalar", where
                    continue
                if dtype != ga.BF16 or mode == "native":
                    # warp rows and the bulk-copy kernels are plain bf16 only
                    assert v in ("cta_row", "split_rows", "scalar"), where
                if v in ("tma_rows", "pipe_rows"):
                    cover = (nt - (32 if v == "pipe_rows" else 0)) * p["vec_per_thread"]
                    assert cover >= nvec, where
                    assert grid <= min(T, GB300_SMS * p["ctas_per_sm"]), where
                    assert p["smem_bytes"] * p["ctas_per_sm"] <= 228 * 1024, where
                    assert p["dynamic_rows"] in (0, 1), where
                else:
                    assert p["dynamic_rows"] == 0 and p["smem_bytes"] == 0, where
                if v == "split_rows":
                    assert p["cluster"] in (2, 4, 8) and grid == T * p["cluster"], where
                    assert grid <= GB300_SMS and nt * p["vec_per_thread"] >= nvec, where
                elif v == "cta_row":
                    sv = -(-nvec // p["cluster"])
                    assert p["cluster"] in (1, 2, 4, 8), where
                    assert nt * p["vec_per_thread"] >= sv, where
                    assert grid == T * p["cluster"], where
                elif v == "warp_rows":
                    assert 32 * p["vec_per_thread"] >= nvec, where
                    assert grid * p["rows_per_cta"] >= T, where
                elif v == "scalar":
                    assert grid == T, where
