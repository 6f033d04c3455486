"""The per-CTA timelines of the tensor-core GEMM and attention kernels
(oases_debug_gemm_timeline, oases_debug_attention_timeline) as the timeline
module reads them: every CTA records its stamps in order, and switching the
timeline off leaves later launches unrecorded."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_gemm_stamps_are_ordered():
    from tensor_model_transformer_tp_gb300 import timeline
    r = timeline.gemm(512, 1024, 512, 2)
    st = r["stamps"]
    assert r["ctas"] > 0 and r["event_us"] > 0
    order = ["entry", "prologue done", "first stage landed", "tile 0 MMAs done", "tile 0 epilogue done",
             "exit"]
    med = [st[k][1] for k in order]
    assert all(a <= b for a, b in zip(med, med[1:])), med
    assert st["tile 0 epilogue done"][3] == r["ctas"]   # every CTA's epilogue stamped


def test_attention_backward_blocks_are_ordered():
    from tensor_model_transformer_tp_gb300 import timeline
    r = timeline.attention_bwd(1, 512, 2)
    for name in ("dq", "dkv"):
        k = r["kernels"][name]
        assert k["span_us"] > 0 and k["cta_mean_us"] > 0
        blocks = np.array(k["cta0_blocks_ns"])
        assert len(blocks) >= 1
        # per block: S/dP issued before the element-wise warp saw S, which is
        # before it handed its dS over
        assert np.all(blocks[:, 2] <= blocks[:, 3])
        # the S/dP MMAs of successive blocks are issued in order
        assert np.all(np.diff(blocks[:, 0]) > 0)


def test_attention_forward_item_stamps_are_ordered():
    from tensor_model_transformer_tp_gb300 import timeline
    r = timeline.attention_fwd(2, 640, 2)   # three tile pairs, the first (heaviest) one ragged
    st = r["stamps"]
    assert r["items"] == 2 * 2 * 3 and r["span_us"] > 0
    for name in ("entry", "set up", "Q and K_0 landed", "tile 0 saw S_0(0)", "tile 0 last PV done",
                 "exit"):
        assert st[name][3] == r["items"], name   # every item stamped
    order = ["entry", "set up", "Q and K_0 landed", "tile 0 saw S_0(0)", "tile 0 last PV done", "exit"]
    med = [st[k][1] for k in order]
    assert all(a <= b for a, b in zip(med, med[1:])), med
    # the pair of tiles 4 and 5 (queries 512..639) has no tile 1: no stamps 5, 6 there
    assert st["tile 1 last PV done"][3] == 2 * 2 * 2


def test_attention_forward_persistent_items_in_order():
    """More items than SMs: every CTA runs its items one after another."""
    from tensor_model_transformer_tp_gb300 import timeline
    r = timeline.attention_fwd(4, 2048, 20)   # 640 items
    assert r["items"] == 640 and 0 < r["ctas"] < 640
    assert 300 < r["sm_mhz"] < 3000   # CTA 0's clock64 over globaltimer
    st = r["stamps"]
    assert st["tile 1 O stored"][3] == 640 and st["exit"][3] == 640
    # heavier pairs take longer
    life = [x[1] for x in r["by_pair"]]
    assert life[0] > life[-1]
