"""Resuming an interrupted configuration sweep (host logic only, no GPU): the
rows already in the output file are recognised by shape, backend and launch
configuration whatever the key order, a line cut short is ignored, and the
appended rows start on a fresh line."""
import json

from skinny_bf16_gemm_residual_gb300 import sweep


def test_row_key_ignores_dict_order():
    a = sweep.row_key(4, 7168, 3584, "rows", {"path": 3, "stages": 3, "k_blocks_per_stage": 8})
    b = sweep.row_key(4, 7168, 3584, "rows", {"k_blocks_per_stage": 8, "path": 3, "stages": 3})
    assert a == b
    assert a != sweep.row_key(8, 7168, 3584, "rows", {"path": 3, "stages": 3, "k_blocks_per_stage": 8})
    assert a != sweep.row_key(4, 7168, 3584, "tile", {"path": 3, "stages": 3, "k_blocks_per_stage": 8})


def test_resume_skips_done_rows_and_repairs_a_cut_line(tmp_path):
    path = tmp_path / "sweep.jsonl"
    done_rows = [
        {"m": 1, "n": 7168, "k": 3584, "backend": "cublas_addmm", "config": {}, "median_us": 12.3},
        {"m": 1, "n": 7168, "k": 3584, "backend": "rows", "config": {"path": 3, "stages": 3}, "median_us": 10.8},
        {"m": 1, "n": 7168, "k": 3584, "backend": "tile", "config": {"path": 4, "tile_n": 512},
         "valid": False, "error": "unsupported"},
    ]
    text = "".join(json.dumps(r) + "\n" for r in done_rows) + '{"m": 2, "n": 7168, "k": 35'  # interrupted write
    path.write_text(text)
    done = sweep.load_done(str(path))
    assert done == {sweep.row_key(r["m"], r["n"], r["k"], r["backend"], r["config"]) for r in done_rows}
    assert sweep.row_key(1, 7168, 3584, "rows", {"stages": 3, "path": 3}) in done
    assert sweep.row_key(2, 7168, 3584, "rows", {"path": 3, "stages": 3}) not in done

    with sweep.open_output(str(path), resume=True) as out:
        out.write(json.dumps({"m": 2, "n": 7168, "k": 3584, "backend": "rows", "config": {}}) + "\n")
    lines = path.read_text().splitlines()
    assert lines[:3] == [json.dumps(r) for r in done_rows]
    assert lines[3] == '{"m": 2, "n": 7168, "k": 35'  # the cut line stays on its own
    assert json.loads(lines[4])["m"] == 2
    assert len(sweep.load_done(str(path))) == 4


def test_fresh_output_and_missing_file(tmp_path):
    path = tmp_path / "new.jsonl"
    assert sweep.load_done(str(path)) == set()
    with sweep.open_output(str(path), resume=True) as out:  # resuming with no file starts one
        out.write("{}\n")
    assert path.read_text() == "{}\n"
    with sweep.open_output(str(path), resume=False) as out:  # a fresh sweep truncates
        out.write("")
    assert path.read_text() == ""


def test_row_metrics():
    peaks = {"hbm_gbs": 6772.9, "bf16_tflops": 1900.0}
    samples = [10.0, 11.0, 12.0]
    r = sweep.build_row(4, 7168, 3584, "rows", {"path": 3}, 4, {"device": "x"}, samples, peaks, "measured")
    nbytes = 2 * (7168 * 3584 + 4 * 3584 + 2 * 4 * 7168)
    assert r["median_us"] == 11.0 and r["device"] == "x" and r["num_buffers"] == 4
    assert abs(r["gbs"] - nbytes / 11e-6 / 1e9) < 1e-9
    assert abs(r["tflops"] - 2 * 4 * 7168 * 3584 / 11e-6 / 1e12) < 1e-9
    assert abs(r["frac_of_hbm_peak"] - r["gbs"] / 6772.9) < 1e-12
    assert abs(r["frac_of_tensor_peak"] - r["tflops"] / 1900.0) < 1e-12
    w = sweep.build_row(4, 7168, 3584, "w8", {"path": 5}, 8, {}, samples, peaks, "measured")
    assert abs(w["gbs"] - (7168 * 3584 + 4 * 7168 + 2 * 4 * 3584 + 4 * 4 * 7168) / 11e-6 / 1e9) < 1e-9
    e = sweep.build_row(4, 7168, 3584, "tile", {"path": 4}, 4, {}, "status 5", peaks, "measured")
    assert e["valid"] is False and e["error"] == "status 5" and "gbs" not in e


def test_peaks_file(tmp_path):
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"hbm_gbs": 6772.9, "bf16_tflops": 1900}))
    assert sweep.load_peaks(str(p)) == ({"hbm_gbs": 6772.9, "bf16_tflops": 1900.0}, "measured")
    assert sweep.load_peaks(str(tmp_path / "absent.json"))[1] == "fallback"
