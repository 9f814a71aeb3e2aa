"""The workspace-free init-routing entry point, for callers that cannot allocate
device memory (a serving engine whose memory pool owns the whole GPU, a
latency-critical loop that must not pay cudaMalloc's synchronisation, a C host
program without a device allocator).  Its scratch is a fixed array inside the
library, so it is compared here, through the C ABI, with the workspace-based
moe_init_routing on two calls in a row (the second call must not see anything
the first left in the shared array).  Collected last on purpose."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


def _same(a: dict, b: dict):
    for key in ("tokens_per_expert", "expert_offsets", "expanded_row_idx", "expanded_x"):
        assert torch.equal(a[key], b[key]), key


def test_noalloc_matches_workspace_version_twice():
    cases = [(4096, 8, 256, 7168, torch.bfloat16, 1), (777, 3, 5, 40, torch.float32, 2)]
    for T, k, E, H, dtype, seed in cases:  # two calls in a row, different shapes and contents
        ids = inputs.random_ids(T, k, E, seed=seed, distinct=(E >= k)).to(DEV)
        x = inputs.random_rows(T, H, dtype, seed=seed, tag="x").to(DEV)
        got = binding.moe_init_routing_noalloc(x, ids, E)
        want = binding.moe_init_routing(x, ids, E)
        torch.cuda.synchronize()
        _same(got, want)
        assert int(got["tokens_per_expert"].sum()) == T * k


def test_noalloc_rejects_requests_beyond_its_scratch():
    T, k, E, H = 200000, 8, 256, 8  # ceil(T*k/1024)*E = 400128 ints > 262144
    x = torch.zeros((1, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((1, k), dtype=torch.int32, device=DEV)
    out = torch.empty(16, dtype=torch.int32, device=DEV)
    st = binding.lib().moe_init_routing_noalloc(binding._ptr(x), binding.MOE_BF16, binding._ptr(ids), T, H, E, k,
                                                binding._ptr(out), binding._ptr(out), binding._ptr(out),
                                                binding._ptr(out), binding._stream())
    assert st == binding.MOE_ERR_UNSUPPORTED


def test_noalloc_bad_ids_match_workspace_version():
    """Ids outside [0,E): not counted, expanded_row_idx = -1, the same outputs as the
    workspace version (whose status word flags them) on the rows both write."""
    T, k, E, H = 300, 4, 16, 64
    ids = inputs.random_ids(T, k, E, seed=31)
    ids[7, 2] = -1
    ids[100, 0] = E
    ids[299, 3] = E + 40
    ids = ids.to(DEV)
    x = inputs.random_rows(T, H, torch.bfloat16, seed=32, tag="x").to(DEV)
    for _ in range(2):
        got = binding.moe_init_routing_noalloc(x, ids, E)
        want = binding.moe_init_routing(x, ids, E)
        assert binding.moe_check_device_status(want["ws"]) & binding.MOE_DEVERR_BAD_EXPERT_ID
        for key in ("tokens_per_expert", "expert_offsets", "expanded_row_idx"):
            assert torch.equal(got[key], want[key]), key
        idx = got["expanded_row_idx"].cpu()
        assert idx[7 * k + 2] == -1 and idx[100 * k] == -1 and idx[299 * k + 3] == -1
        assert int(got["tokens_per_expert"].sum()) == T * k - 3
        n = int(got["expert_offsets"][E])
        assert n == T * k - 3
        assert torch.equal(got["expanded_x"][:n], want["expanded_x"][:n])


def test_noalloc_empty_batch_writes_zero_counts():
    """T = 0: every count and offset is written as 0, whatever the buffers held."""
    E, k, H = 40, 3, 16
    x = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((0, k), dtype=torch.int32, device=DEV)
    for _ in range(2):
        counts = torch.full((E,), 7, dtype=torch.int32, device=DEV)
        offsets = torch.full((E + 1,), 7, dtype=torch.int32, device=DEV)
        st = binding.lib().moe_init_routing_noalloc(binding._ptr(x), binding.MOE_BF16, binding._ptr(ids), 0, H, E,
                                                    k, None, None, binding._ptr(counts), binding._ptr(offsets),
                                                    binding._stream())
        assert st == binding.MOE_OK
        torch.cuda.synchronize()
        assert torch.all(counts == 0) and torch.all(offsets == 0)
