"""The single-shape command-line tool on the GPU (small shapes, one call each)."""

import pytest

from tensor_comm_gemm_gb300 import run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("argv,shape", [
    (["--op", "ag", "--tp", "2", "--n", "256", "--k", "256", "--m", "256"], "cta_group 1"),
    (["--op", "ag", "--tp", "2", "--n", "512", "--k", "256", "--m", "512", "--dtype", "e4m3"], "cta_group 2"),
    (["--op", "rs", "--tp", "4", "--n", "1024", "--k", "512", "--m", "256"], "cta_group 2"),
    (["--op", "ar", "--tp", "2", "--n", "1024", "--k", "256", "--m", "256", "--chunks", "2"], "cta_group 2"),
])
def test_run_case_reports_time_and_launch_shape(capsys, argv, shape):
    run_case.main(argv + ["--calls", "2"])
    out = capsys.readouterr().out
    assert "TFLOP/s" in out and shape in out, out
