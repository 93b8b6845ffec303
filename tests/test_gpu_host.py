"""Host-buffer entry points: HostRunner (one step) and HostPipeline (steps
whose copies overlap their neighbours' kernels) return what the device-side
calls return on the same inputs (bit for bit, except dQ's last place)."""

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tiled_attention_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def device_reference(q, k, v, do, causal):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal)
    dq, dk, dv, _ = fa.attention_backward(qd, kd, vd, o, lse, dod, causal)
    torch.cuda.synchronize()
    return {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


def same(got, ref):
    # O, LSE, dK, dV are formed in a fixed order and match bit for bit.  dQ is
    # summed in fp32 by reductions from many CTAs in hardware order before its
    # 16-bit rounding, so it may differ by one unit in the last place.
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(got[name], ref[name]), name
    a, b = got["dq"].double(), ref["dq"].double()
    assert torch.all((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-6), "dq"


@pytest.mark.parametrize("causal", [False, True])
def test_host_runner_matches_device_calls(cuda_lib, causal):
    B, L, H, Hkv, D = 2, 300, 4, 2, 128
    q, k, v, do = make_qkv(B, L, H, Hkv, D, "bf16", seed=11)
    runner = fa.HostRunner(B, L, H, Hkv, D, torch.bfloat16, causal)
    out = runner.run(*(x.pin_memory() for x in (q, k, v, do)))
    torch.cuda.synchronize()
    same(out, device_reference(q, k, v, do, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_host_pipeline_matches_device_calls(cuda_lib, causal):
    B, L, H, Hkv, D = 2, 257, 4, 1, 64
    runner = fa.HostPipeline(B, L, H, Hkv, D, torch.float16, causal, depth=2)
    batches = [make_qkv(B, L, H, Hkv, D, "fp16", seed=20 + s) for s in range(5)]
    refs = [device_reference(*b, causal) for b in batches]
    pinned = [tuple(x.pin_memory() for x in b) for b in batches]
    # two steps in flight, then read them; then three more (sets reused)
    outs = [runner.submit(*pinned[0]), runner.submit(*pinned[1])]
    runner.wait()
    for s in range(2):
        same(outs[s], refs[s])
    for s in range(2, 5):
        out = runner.submit(*pinned[s])
    runner.wait()
    same(out, refs[4])
    assert runner.h2d_bytes() == 2 * (2 * B * L * H * D + 2 * B * L * Hkv * D)
