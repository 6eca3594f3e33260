"""The verify step's accepted-draft count and bonus token against the oracle:
integer work, so bit-exact, over block sizes that use one, two and three
32-position rounds of the warp ballot, strided rows and a block of one."""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from draft_model_kv_gb300 import build
    build.build()


@pytest.mark.parametrize("batch,block", [(64, 8), (4096, 8), (1000, 16), (7, 1), (33, 33), (300, 70), (1, 2)])
def test_matches_oracle(batch, block):
    import draft_model_kv_gb300 as dk
    cand, tgt = synthetic.make_verify_workload(batch, block, seed=batch + block)
    correct, bonus = dk.dspark_correct_drafts_and_bonus(torch.from_numpy(cand).cuda(), torch.from_numpy(tgt).cuda())
    torch.cuda.synchronize()
    rc, rb = oracle.correct_drafts_and_bonus(cand, tgt)
    np.testing.assert_array_equal(correct.cpu().numpy(), rc)
    np.testing.assert_array_equal(bonus.cpu().numpy(), rb)


def test_strided_rows_and_empty_batch():
    import draft_model_kv_gb300 as dk
    cand, tgt = synthetic.make_verify_workload(50, 12, seed=3)
    wide_c = torch.zeros((50, 20), dtype=torch.int64, device="cuda")
    wide_t = torch.full((50, 17), -5, dtype=torch.int64, device="cuda")
    wide_c[:, :12] = torch.from_numpy(cand).cuda()
    wide_t[:, :12] = torch.from_numpy(tgt).cuda()
    correct, bonus = dk.dspark_correct_drafts_and_bonus(wide_c[:, :12], wide_t[:, :12])
    torch.cuda.synchronize()
    rc, rb = oracle.correct_drafts_and_bonus(cand, tgt)
    np.testing.assert_array_equal(correct.cpu().numpy(), rc)
    np.testing.assert_array_equal(bonus.cpu().numpy(), rb)
    e = torch.empty((0, 8), dtype=torch.int64, device="cuda")
    c0, b0 = dk.dspark_correct_drafts_and_bonus(e, e)
    assert c0.numel() == 0 and b0.numel() == 0
