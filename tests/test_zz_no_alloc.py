"""lmoe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (no handle, scratch in a static device array).

Checked through the C ABI against the handle-based lmoe_dispatch, bit for
bit, on two calls in a row (the second at the maximum size, after the first
left its contents in the shared scratch); sizes beyond the maximum are
rejected before any launch.  Collected last so that a run stopping at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

from lmoe_inputs import configs as C
from tests._harness import gpu_inputs, make_layer

pytestmark = pytest.mark.gpu


def _idx(T, k, E, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32))


def test_noalloc_dispatch_matches_handle_dispatch():
    from latent_mixture_experts_gb300 import binding
    wl = C.workload("k3_tiny_t16")
    E, k = wl.cfg.n_experts, wl.cfg.top_k
    T_max = binding.NOALLOC_MAX_ASSIGNMENTS // k
    W, _ = gpu_inputs(wl, T=1)
    layer = make_layer(wl, W, max_tokens=T_max)
    for call, (T, seed) in enumerate(((1000, 11), (T_max, 12))):
        idx = _idx(T, k, E, seed).cuda()
        want = [t.cpu() for t in layer.lmoe_dispatch(idx)]
        counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
        perm = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
        binding.lmoe_dispatch_noalloc(idx, E, counts, offsets, perm)
        torch.cuda.synchronize()
        for got, ref in zip((counts, offsets, perm), want):
            assert torch.equal(got.cpu(), ref), f"call {call}"
    layer.lmoe_sync_status()
    layer.close()


@pytest.mark.parametrize("E,k,P", [(2048, 8, 8192), (2048, 8, 65536), (896, 16, 65536), (896, 16, 1024)],
                         ids=["E2048_one_block", "E2048_max", "k3_max", "k3_t64"])
def test_noalloc_dispatch_at_the_limits(E, k, P):
    """Sizes at the documented limits (2048 experts; 65,536 assignments, the
    largest batch; 8,192, the largest the one-kernel dispatch takes) and the
    Kimi-K3 routing shape, bit for bit against the oracle's counting sort."""
    import oracle as O
    from latent_mixture_experts_gb300 import binding
    T = P // k
    idx = _idx(T, k, E, seed=P + E).cuda()
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((P,), -1, dtype=torch.int32, device="cuda")
    binding.lmoe_dispatch_noalloc(idx, E, counts, offsets, perm)
    torch.cuda.synchronize()
    d = O.dispatch(idx.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), d["counts"])
    assert np.array_equal(offsets.cpu().numpy(), d["offsets"])
    assert np.array_equal(perm.cpu().numpy(), d["perm"])


def test_noalloc_dispatch_rejects_oversize():
    from latent_mixture_experts_gb300 import binding
    from latent_mixture_experts_gb300 import LmoeError, LMOE_ERR_INVALID_ARG
    k = 2
    T = binding.NOALLOC_MAX_ASSIGNMENTS // k + 1
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    out = torch.empty(T * k + 2 * binding.NOALLOC_MAX_EXPERTS + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(LmoeError) as ei:
        binding.lmoe_dispatch_noalloc(idx, 64, out, out, out)
    assert ei.value.status == LMOE_ERR_INVALID_ARG
    idx = torch.zeros(4, k, dtype=torch.int32, device="cuda")
    with pytest.raises(LmoeError):
        binding.lmoe_dispatch_noalloc(idx, binding.NOALLOC_MAX_EXPERTS + 1, out, out, out)
