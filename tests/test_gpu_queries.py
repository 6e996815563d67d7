"""The host queries that need a device: default configurations per path and
the resources of the kernel each path launches (registers, spills, shared
memory, threads), like the register/spill query of the benchmark page."""
import pytest
import torch

import skinny_bf16_gemm_residual_gb300 as sgr

pytestmark = pytest.mark.gpu

N, K = 7168, 3584


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    sgr.sgr_init(0)


@pytest.mark.parametrize("M", [1, 4, 16, 64, 256, 1024])
def test_default_config_auto_matches_selected_path(M):
    c = sgr.sgr_default_config(M, N, K)
    assert c.path == sgr.sgr_select_path(M, N, K)
    assert c.stages >= 1 and c.ctas_per_sm >= 1


# local (stack) bytes per thread: none, except a 16-byte local array in the
# stream-K kernel (no register spills anywhere).
@pytest.mark.parametrize("path,M,threads,local", [
    (sgr.SGR_PATH_TC_ROWS, 4, 224, 0), (sgr.SGR_PATH_TILE, 1024, 192, 0), (sgr.SGR_PATH_SIMT, 4, 256, 0),
    (sgr.SGR_PATH_TC, 8, None, 16), (sgr.SGR_PATH_W8, 4, 352, 0)])
def test_kernel_resources(path, M, threads, local):
    r = sgr.sgr_kernel_resources(M, N, K, path=path)
    assert 0 < r["registers_per_thread"] <= 255
    assert r["spill_bytes"] <= local, r
    assert r["smem_bytes"] <= 232448
    if threads is not None:
        assert r["threads"] == threads
    assert r["registers_per_thread"] * r["threads"] <= 65536
    if path == sgr.SGR_PATH_TC_ROWS:  # two CTAs per SM where shared memory allows
        assert 2 * r["registers_per_thread"] * r["threads"] <= 65536


def test_fp8_default_config():
    c = sgr.sgr_default_config(4, N, K, path=sgr.SGR_PATH_W8)
    assert (c.path, c.k_blocks_per_stage, c.stages, c.prefetch_stages, c.token_tile) == (sgr.SGR_PATH_W8, 8, 2, 2, 16)
    r = sgr.sgr_kernel_resources(4, N, K, path=sgr.SGR_PATH_W8)
    assert 2 * (r["smem_bytes"] + 1024) <= 233472, "two CTAs per SM must fit"
    assert 2 * r["registers_per_thread"] * r["threads"] <= 65536


def test_queries_reject_bad_shapes():
    with pytest.raises(sgr.SgrError):
        sgr.sgr_default_config(4, 7170, K)
    with pytest.raises(sgr.SgrError):
        sgr.sgr_kernel_resources(0, N, K)


def table_entries(n: int, k: int):
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "skinny_bf16_gemm_residual_gb300", "csrc", "sgr_table.h")
    rows = []
    for m in re.finditer(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+),",
                         open(path).read()):
        v = [int(x) for x in m.groups()]
        if v[0] == n and v[1] == k:
            rows.append(dict(m=v[2], path=v[3], ctas_per_sm=v[4], stages=v[5], rows_per_stage=v[6],
                             k_blocks_per_stage=v[7], prefetch_stages=v[8], tile_n=v[9], k_split=v[10]))
    return rows


@pytest.mark.parametrize("n,k", [(7168, 3584), (3584, 7168)])
def test_automatic_config_is_the_measured_table_entry(n, k):
    """Every field the table holds for a shape reaches the launch configuration
    the library uses for it (at the table's own M)."""
    entries = table_entries(n, k)
    assert entries
    for e in entries:
        c = sgr.sgr_default_config(e["m"], n, k)
        assert c.path == e["path"], e
        assert (c.ctas_per_sm, c.stages) == (e["ctas_per_sm"], e["stages"]), (e, c.as_dict())
        if e["path"] != sgr.SGR_PATH_SIMT and (e["path"] != sgr.SGR_PATH_TILE or e["k_blocks_per_stage"] > 0):
            assert c.k_blocks_per_stage == e["k_blocks_per_stage"], (e, c.as_dict())
        if e["path"] in (sgr.SGR_PATH_TC_ROWS, sgr.SGR_PATH_SIMT):
            assert c.rows_per_stage == e["rows_per_stage"], (e, c.as_dict())
        if e["path"] in (sgr.SGR_PATH_TC_ROWS, sgr.SGR_PATH_TILE, sgr.SGR_PATH_PAIR):
            assert c.prefetch_stages == e["prefetch_stages"], (e, c.as_dict())
        if e["path"] == sgr.SGR_PATH_TILE:
            assert (c.tile_n, c.k_split) == (e["tile_n"], max(e["k_split"], 1)), (e, c.as_dict())
        if e["path"] == sgr.SGR_PATH_PAIR:
            assert c.tile_n == e["tile_n"], (e, c.as_dict())
