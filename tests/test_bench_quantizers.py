"""bench.py's per-kernel quantizer records, from a made-up trace: each
quantizer launch is matched to its algorithmic bytes by kernel name (a name
that repeats is taken in turn, a trailing * matches a prefix), the first
alternative whose kernels all appear in a step is the one used, and the
span runs from the first quantizer's start to the last one's end."""
import pytest

from tests.conftest import ROOT  # noqa: F401  (puts the repo root on sys.path)


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def _work(bench, want):
    class Fake(bench.Work):
        def quantizer_bytes(self):
            return want
    return Fake()


def test_alternatives_names_and_span(bench):
    G = 10**9
    want = [[("dual", "qdual", G), ("pair", "qpair", 3 * G)],
            [("dual", "qdual", G), ("w", "qcol", G), ("x", "qcol", 2 * G)]]
    # two steps of the second form: each step the dual then two column launches, then a GEMM
    launches = []
    for st in range(2):
        t = 10.0 * st
        launches += [("qdual", t + 0.0, 1.0), ("qcol", t + 1.0, 0.5), ("qcol", t + 1.5, 1.0), ("gemm", t + 2.5, 5.0)]
    rep = _work(bench, want).quantizer_report(launches, 2)
    assert set(rep) == {"dual", "w", "x", "all quantizers, first start to last end"}
    assert rep["dual"]["gbs"] == pytest.approx(1000.0)   # 1 GB in 1 ms
    assert rep["w"]["gbs"] == pytest.approx(2000.0)      # the step's first qcol: 1 GB in 0.5 ms
    assert rep["x"]["gbs"] == pytest.approx(2000.0)      # its second: 2 GB in 1 ms
    assert rep["x"]["us_per_step"] == pytest.approx(1000.0)
    span = rep["all quantizers, first start to last end"]
    assert span["us_per_step"] == pytest.approx(2500.0)                  # 0 .. 2.5 ms each step
    assert span["bytes_per_step"] == 4 * G
    assert span["gbs"] == pytest.approx(1600.0)          # 4 GB in 2.5 ms


def test_prefix_match_and_first_alternative(bench):
    want = [[("rows", "quant_rows*", 4 * 10**8), ("tiles", "quant_tile_batch", 8 * 10**8)]]
    launches = [("quant_tile_batch", 0.0, 2.0), ("quant_rows_reg", 2.0, 1.0), ("gemm", 3.0, 4.0)]
    rep = _work(bench, want).quantizer_report(launches, 1)
    assert rep["rows"]["kernel"] == "quant_rows_reg"
    assert rep["tiles"]["gbs"] == pytest.approx(400.0)   # 0.8 GB in 2 ms
    assert rep["all quantizers, first start to last end"]["us_per_step"] == pytest.approx(3000.0)
