"""The grouped GEMMs' stage timing (a measurement aid of the diagnostic build): armed for
one kind, that kind's next launch stamps CTA 0's pipeline stages and tiles in order; an
armed launch computes exactly what an unarmed one does; disarmed, nothing is stamped.
The diagnostic library replaces the shipped one for a whole process, so the check runs
as its own process. The shipped library refuses the calls."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    assert torch.cuda.is_available()
    return m


def test_diagnostic_build_stamps_in_order_and_changes_nothing():
    r = subprocess.run([sys.executable, "-m", "moe_expert_layer_route_gb300.stage_timing",
                        "--check"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "stage timing check ok" in r.stdout


def test_shipped_library_has_no_stage_timing(moe):
    with pytest.raises(moe.MoEError) as ex:
        moe.stage_timing_arm("down")
    assert ex.value.status == -2                  # MOE_ERR_UNSUPPORTED
