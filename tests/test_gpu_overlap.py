"""The prefill kernel's two schedules (side stream beside the decode kernel,
or serial on the caller's stream) give bit-identical results that match the
oracle, and the prefill profile events time the prefill kernel."""
import pytest
import torch

import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

from helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_attention_04_gb300 import build
    build.build()
    P.lib()


def test_serial_and_overlapped_prefill_are_bit_identical():
    spec = W.custom_spec("overlap", "bf16", 32, 8, 128, [1, 1, 1, 300, 64, 1],
                         [900, 2100, 40, 1500, 64, 5000], seed=71)
    cpu = W.make_step(spec)
    st = cpu.to("cuda")
    try:
        P.pa_set_prefill_overlap(False)
        serial, *_, s1 = run_gpu(st)
        P.pa_set_prefill_overlap(True)
        overlapped, *_, s2 = run_gpu(st)
    finally:
        P.pa_set_prefill_overlap(True)
    assert s1 == 0 and s2 == 0
    assert torch.equal(serial.view(torch.int16), overlapped.view(torch.int16))
    ref, _, _ = run_oracle(cpu)
    assert_close(overlapped, ref, "bf16", "overlap case")


@pytest.mark.parametrize("overlap", [True, False])
def test_prefill_profile_events_time_the_prefill_kernel(overlap):
    spec = W.custom_spec("pf-events", "bf16", 32, 8, 128, [512, 1], [2048, 700], seed=72)
    st = W.make_step(spec, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        P.pa_set_prefill_overlap(overlap)
        P.pa_set_prefill_profile_events(a, b)
        run_gpu(st)
    finally:
        P.pa_set_prefill_profile_events(None, None)
        P.pa_set_prefill_overlap(True)
    torch.cuda.synchronize()
    assert a.elapsed_time(b) > 0
