"""The measured tensor-core ceilings the benchmark reports beside the nominal
FP4 peak: they run, leave the status word clean, and relate as measured on
GB300 (the paired MMA a little below the single-CTA one, both below the
nominal 13.5 PFLOP/s dense FP4 figure)."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def test_fp4_mma_ceilings():
    import audio_dit_gb300 as A
    ws = A.alloc_workspace(128, 256, 256, 0)
    single = A.h3fp4_measure_fp4_peak(ws, 4000)
    pair = A.h3fp4_measure_fp4_pair_peak(ws, 4000)
    A.h3fp4_check(ws)
    assert 1000.0 < single < 13500.0
    assert 1000.0 < pair < 13500.0
    assert pair < 1.1 * single
