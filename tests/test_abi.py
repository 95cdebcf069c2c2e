"""The C ABI without a GPU: the library builds and loads, exports every
function include/eg.h declares, and rejects bad problems before touching a
device."""
import ctypes

import pytest
import torch

import epilogue_tcgen05_tmem_gb300 as eg
from epilogue_tcgen05_tmem_gb300 import _build
from tests._gpu_helpers import header_functions


@pytest.fixture(scope="module")
def L():
    _build.build()
    return eg.lib()


def test_exports_every_declared_function(L):
    names = header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(eg.EXPORTED)


def test_status_strings(L):
    for s in range(7):
        assert eg.status_string(s).startswith("EG_")
    assert eg.status_string(99) == "EG_ERR_UNKNOWN"


BAD = [
    (dict(M=-1, N=8, K=64), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="bf16", scale="token_channel"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="e4m3", scale="none"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="int8", scale="block"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=192, dtype="e4m3", scale="block"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=60), eg.EG_ERR_INVALID_ARG),            # 120 bytes: not 16-aligned
    (dict(M=4, N=8, K=136, dtype="e4m3", scale="token_channel"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=133152, dtype="int8", scale="token_channel"), eg.EG_ERR_UNSUPPORTED),
    (dict(M=4, N=8, K=64, flags=eg.EG_EPI_RESIDUAL | eg.EG_EPI_RESIDUAL_PRE_ACT), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, flags=1 << 12), eg.EG_ERR_INVALID_ARG),
    # gated units: block scales need the up half on a weight block; no
    # pre-activation residual, no accumulator output
    (dict(M=4, N=200, K=256, dtype="e4m3", scale="block", flags=eg.EG_EPI_GATED), eg.EG_ERR_UNSUPPORTED),
    (dict(M=4, N=256, K=256, dtype="int8", scale="token_channel",
          flags=eg.EG_EPI_GATED | eg.EG_EPI_RESIDUAL_PRE_ACT), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=256, K=256, dtype="e4m3", scale="block",
          flags=eg.EG_EPI_GATED | eg.EG_OUT_DEBUG_ACCUM), eg.EG_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("kw,status", BAD)
def test_invalid_problems_rejected_before_device(L, kw, status):
    kw = dict(kw)
    flags = kw.pop("flags", 0)
    p = eg.make_problem(flags=flags, **kw)
    s, h = eg.eg_plan_create(p)
    assert s == status and h is None
    assert eg.last_error_detail()


def test_invalid_activation(L):
    p = eg.make_problem(4, 8, 64)
    p.act = 9
    s, _ = eg.eg_plan_create(p)
    assert s == eg.EG_ERR_INVALID_ARG


def test_null_arguments(L):
    assert L.eg_plan_create(None, None, None) == eg.EG_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.eg_plan_create(None, None, ctypes.byref(h)) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_destroy(None) == eg.EG_OK
    assert L.eg_plan_run(None, None, None) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_device_status(None) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_last_launch_count(None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_problem_without_device_reports_cuda_error(L):
    s, h = eg.eg_plan_create(eg.make_problem(4, 8, 64))
    assert s == eg.EG_ERR_CUDA and h is None
    assert "cuda" in eg.last_error_detail().lower()


def test_plan_class_raises_loudly(L):
    with pytest.raises(eg.EgError):
        eg.Plan(-1, 8, 64)


def _c_struct_fields(name):
    """Field names of a typedef struct in include/eg.h, in order."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "eg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*" + name + ";", src).group(1)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            fields += [f.strip().lstrip("*") for f in decl.split(None, 1)[1].split(",")]
    return fields


@pytest.mark.parametrize("name,cls", [("eg_tuning", eg.eg_tuning), ("eg_problem", eg.eg_problem)])
def test_binding_structs_match_header(name, cls):
    assert [f for f, _ in cls._fields_] == _c_struct_fields(name)


def test_tuning_table_rows_are_valid():
    """Every swept row has the 13 fields of the table, an epilogue class of
    0, 1 or 2, uses the cluster reduction only with a split of 2, 4 or 8 and
    without balanced split-K, CTA pairs only unsplit, without swap-AB, with
    tiles of 128 or 256, and gated rows only the gated kernels' tiles."""
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "epilogue_tcgen05_tmem_gb300", "csrc", "eg_tuning_table.inc")
    rows = [tuple(int(x) for x in m.split(","))
            for m in re.findall(r"^\s*\{([-\d, ]+)\},", open(path).read(), flags=re.M)]
    assert rows
    for r in rows:
        assert len(r) == 13, r
        dtype, scale, N, K, bucket, epi, tn, stages, split, swap, sk, cl, pair = r
        assert epi in (0, 1, 2), r
        if epi == 1:
            assert tn in ((16, 32, 64) if swap else (64, 128)) and cl == 0 and pair == 0, r
        assert bucket in (0, 1, 2, 4, 8, 16, 24, 32, 64, 128, 256, 512, 1024, 2048)
        assert tn in (16, 32, 64, 128, 192, 224, 256)
        if tn in (192, 224):
            assert swap == 0 and scale != 2 and dtype != 2, r
        assert 2 <= stages <= 8 and swap in (0, 1) and cl in (0, 1)
        if cl:
            assert split in (2, 4, 8) and sk == 0, r
        if sk:
            assert split == 1, r
        assert pair in (0, 1)
        if pair:
            assert split == 1 and sk == 0 and cl == 0 and swap == 0 and tn in (128, 256), r
            assert scale != 2 and dtype != 2, r


def test_sweep_candidates_and_rows():
    from epilogue_tcgen05_tmem_gb300 import inputs, sweep
    p = inputs.make_problem(16, 1024, 4096, "e4m3", "token_channel", seed=0)
    cands = list(sweep.candidates(p, swaps=(1,)))
    keys = {"tile_n", "stages", "split_k", "swap_ab", "stream_k", "cluster_reduce", "cta_pair"}
    assert all(set(c) == keys for c in cands)
    cl = [c for c in cands if c["cluster_reduce"]]
    assert cl and all(c["split_k"] in (2, 4, 8) and c["stream_k"] == 0 for c in cl)
    text = sweep.format_rows([(1, 1, 1024, 4096, 16, 0, 16, 4, 4, 1, 0, 1, 0)])
    assert text.strip() == "{1, 1, 1024, 4096, 16, 0, 16, 4, 4, 1, 0, 1, 0},"


def test_sweep_gated_candidates_use_gated_kernels():
    from epilogue_tcgen05_tmem_gb300 import sweep
    p, epi = sweep.sweep_problem("fp8_swiglu", 8)
    assert epi == sweep.EPI_GATED and p.meta.get("gated") and p.W.shape[0] == 2 * p.N
    cands = [c for c in sweep.candidates(p, swaps=(0, 1)) if sweep.gated_ok(c)]
    assert cands and all(c["tile_n"] in sweep.GATED_TILES[c["swap_ab"]] for c in cands)
    q, e = sweep.sweep_problem("int8_quant", 4)
    assert e == sweep.EPI_QUANT and q.dtype == "int8"


def test_sweep_pair_candidates():
    """Above the decode buckets the sweep also tries CTA pairs, only where the
    pair kernels exist: no swap-AB, per-token/channel or bf16, unsplit."""
    from epilogue_tcgen05_tmem_gb300 import inputs, sweep
    p = inputs.make_problem(256, 512, 256, "e4m3", "token_channel", seed=0)
    cands = list(sweep.candidates(p, swaps=(0, 1)))
    pairs = [c for c in cands if c["cta_pair"]]
    assert pairs
    assert all(c["swap_ab"] == 0 and c["split_k"] == 1 and c["stream_k"] == 0
               and c["cluster_reduce"] == 0 and c["tile_n"] in (128, 256) for c in pairs)
    pb = inputs.make_problem(256, 512, 256, "e4m3", "block", seed=0)
    assert not [c for c in sweep.candidates(pb, swaps=(0,)) if c["cta_pair"]]


def test_sweep_block_wide_tiles_only_over_m():
    """Block-scale tiles 256 wide exist with rows over M only."""
    from epilogue_tcgen05_tmem_gb300 import inputs, sweep
    pb = inputs.make_problem(512, 1024, 512, "e4m3", "block", seed=0)
    cands = list(sweep.candidates(pb, swaps=(0, 1)))
    wide = [c for c in cands if c["tile_n"] > 128]
    assert wide and all(c["swap_ab"] == 0 and c["tile_n"] == 256 for c in wide)
