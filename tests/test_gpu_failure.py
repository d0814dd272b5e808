"""The failure path of the bounded device waits, made to run out on purpose without any
fault: one GEMV launch whose producer issues no copies, so its consumers wait on stages that
never fill, give up after their clock budget and return.  The error word must surface as
FQ_ERR_DEVICE_TIMEOUT from fq_check_device (section 14.2's error-set convention: failures
come back as a status, not as a crash), and the next steps on the same stream must match
the oracle again."""
import pytest

from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import stream
from tests.test_gpu_parity import SMALL, _compare_step, pair_factory, workload  # noqa: F401

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_later_steps_are_correct(pair_factory):  # noqa: F811
    p = pair_factory(workload(SMALL, "q8_0", "bf16", seed=61), max_positions=256)
    kvc, oc = p.new_seq(capacity=128, ctx=40, seq=0)
    _compare_step(p, [kvc], [oc], [5], "before the timeout")
    fq.fq_check_device(p.model, stream())
    fq.fq_debug_wait_timeout(p.model, stream())
    with pytest.raises(fq.FqError) as e:
        fq.fq_check_device(p.model, stream())
    assert e.value.status == fq.DEVICE_TIMEOUT
    fq.fq_check_device(p.model, stream())               # the record was cleared
    for i, tok in enumerate((7, 11)):
        _compare_step(p, [kvc], [oc], [tok], f"step {i} after the timeout")
    fq.fq_check_device(p.model, stream())
    assert fq.fq_kv_len(kvc) == 43
