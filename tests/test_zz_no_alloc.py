"""The allocation-free entry point against the regular split + combine.

fp8kv_attn_forward_static is for callers that cannot allocate device memory
(a host runtime that hands a plugin only its inputs and outputs, a memory
manager that owns the whole heap, a path that forbids allocator calls): it
keeps its FP32 partials in the library's own device array.  Two calls in a
row (the second with other row lengths, so stale partials from the first
would show) must give the regular entry point's output bit for bit (same
plan, same kernels), and a plan whose partials exceed the array is refused.  This file is
collected last so that a stop at the first failure has run every other test.
"""

import pytest
import torch


pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()


def _regular_and_static(dp):
    from fp8_e4m3_paged_gb300 import binding as B

    s = torch.cuda.current_stream().cuda_stream
    dp.out.zero_()
    dp.calls[0].run(s)
    torch.cuda.synchronize()
    regular = dp.out.clone()
    dp.out.fill_(float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    a = B.Args.from_buffer_copy(dp.calls[0].args)
    a.workspace = status.data_ptr()
    a.workspace_bytes = 4
    B.fp8kv_attn_forward_static(dp.plan, a, s)
    torch.cuda.synchronize()
    return regular, dp.out.clone(), int(status.item())


def _same_bits(x, y):
    return torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("name", ["c2", "c3_64k", "c5"])
def test_static_matches_regular_twice(name):
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem
    from synth import make_problem
    from synth.workloads import causal_row_len

    p = make_problem(name)
    dp = DeviceProblem(p)
    assert dp.plan.workspace_bytes <= 16 << 20
    regular, static, status = _regular_and_static(dp)
    assert _same_bits(static, regular), f"{name} static call 1"
    assert status == 0
    if p.mode == "dense":
        # second call with fewer live rows: stale partials would show up here
        dp.row_len.copy_(torch.tensor([causal_row_len(p.max_kv_len, p.q, 3)], dtype=torch.int32))
    else:
        dp.q.mul_(-1.0)
    regular2, static2, status2 = _regular_and_static(dp)
    assert _same_bits(static2, regular2), f"{name} static call 2"
    assert status2 == 0
    assert not _same_bits(regular, regular2)


def test_static_batch_zero_clears_status_word():
    from fp8_e4m3_paged_gb300 import binding as B

    d = B.make_desc(mode=0, batch=0, q_max=1, num_q_heads=1, num_kv_heads=1, head_dim=64,
                    page_size=16, max_kv_len=0, max_blocks=0, num_kv_blocks=1)
    plan = B.fp8kv_attn_plan(d)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    a = B.Args()
    a.workspace = status.data_ptr()
    a.workspace_bytes = 4
    B.fp8kv_attn_forward_static(plan, a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_static_rejects_oversized_plan():
    from fp8_e4m3_paged_gb300 import binding as B

    d = B.make_desc(mode=0, batch=64, q_max=8, num_q_heads=32, num_kv_heads=8, head_dim=256, page_size=16,
                    max_kv_len=65536, max_blocks=4096, num_kv_blocks=1 << 20, num_splits=64)
    plan = B.fp8kv_attn_plan(d)
    assert plan.workspace_bytes > B.STATIC_SCRATCH_BYTES
    a = B.Args()
    with pytest.raises(B.Fp8kvError) as ei:
        B.fp8kv_attn_forward_static(plan, a, torch.cuda.current_stream().cuda_stream)
    assert ei.value.code == B.EWORKSPACE
