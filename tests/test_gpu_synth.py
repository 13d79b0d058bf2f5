"""The CUDA twin of the seeded record generator agrees bit for bit with the
numpy generator (pools of the full-size configurations are built with it)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.mark.parametrize("wd,H,I,keys", [(synth.WD_FP32, 256, 128, [0, 31]),
                                         (synth.WD_BF16, 2048, 512, [0, 10239, 10240 + 39]),
                                         (synth.WD_FP4, 4096, 2048, [5, 11007]),
                                         (synth.WD_FP4, 512, 256, [0, 1, 2, 47])])
def test_gpu_records_match_numpy(wd, H, I, keys):
    S = synth.record_bytes(H, I, wd)
    for key in keys:
        dev = torch.empty(S, dtype=torch.uint8, device="cuda")
        synth.records_gpu(dev.data_ptr(), 3, key, 1, H, I, wd)
        assert (dev.cpu().numpy() == synth.expert_record(3, key, H, I, wd)).all(), (wd, key)


def test_pinned_pool_matches_c_generator():
    pool = synth.pinned_pool(7, 24, 512, 256, synth.WD_FP4, chunk_bytes=3 * synth.record_bytes(512, 256, synth.WD_FP4))
    ref = synth.records_array(7, 0, 24, 512, 256, synth.WD_FP4)
    assert pool.shape == ref.shape and (pool == ref).all()
