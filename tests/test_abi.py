"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any GPU work.
No compute call runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from tests._harness import built_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def declared_functions():
    """Every function any header under include/ declares."""
    names = set()
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            names.update(re.findall(r"^\s*(?:LMOE_API\s+)?(?:lmoe_status|const char\s*\*|int)\s+(lmoe_\w+)\s*\(",
                                    text, re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    built_library()
    from latent_mixture_experts_gb300 import binding
    return binding.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lmoe_create", "lmoe_route", "lmoe_forward", "lmoe_destroy", "lmoe_tc_peak"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from latent_mixture_experts_gb300 import binding
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from latent_mixture_experts_gb300 import binding
    for code in range(6):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"


def _cfg(**kw):
    from latent_mixture_experts_gb300 import binding
    from lmoe_inputs import K3_TINY
    c = binding.make_config(K3_TINY, 16)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _weights(skip=()):
    from latent_mixture_experts_gb300 import binding
    # Aligned, never dereferenced on the host: validation must fail or the
    # device lookup must report CUDA before anything touches them.
    vals = {n: (0 if n in skip else 0x10000 + 256 * i) for i, n in enumerate(binding._WEIGHT_FIELDS)}
    return binding.LmoeWeights(**vals)


def _create(lib, cfg, w, out=True):
    h = ctypes.c_void_p()
    return lib.lmoe_create(ctypes.byref(cfg) if cfg is not None else None,
                           ctypes.byref(w) if w is not None else None, None,
                           ctypes.byref(h) if out else None), h


def test_create_rejects_bad_arguments(lib):
    from latent_mixture_experts_gb300 import binding as b
    assert _create(lib, _cfg(), _weights(), out=False)[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, None, _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(), None)[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(top_k=65), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(max_tokens=0), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(act=7), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(d_latent=336 + 8), _weights())[0] == b.LMOE_ERR_UNSUPPORTED
    assert _create(lib, _cfg(expert_wfmt=1), _weights())[0] == b.LMOE_ERR_UNSUPPORTED
    assert _create(lib, _cfg(n_experts=4096, top_k=2), _weights())[0] == b.LMOE_ERR_UNSUPPORTED
    assert _create(lib, _cfg(), _weights(skip=("ex_up_q",)))[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(), _weights(skip=("norm_w",)))[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(act_terms=3), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(act_format=1, act_terms=5), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(ep_size=3), _weights())[0] == b.LMOE_ERR_INVALID_ARG      # 64 experts over 3 ranks
    assert _create(lib, _cfg(ep_size=2, ep_rank=2), _weights())[0] == b.LMOE_ERR_INVALID_ARG
    assert _create(lib, _cfg(ep_size=2, act_format=1), _weights())[0] == b.LMOE_ERR_UNSUPPORTED
    assert _create(lib, _cfg(act_terms=1, expert_wfmt=1, d_latent=0, use_latent_norm=0),
                   _weights())[0] == b.LMOE_ERR_UNSUPPORTED     # one-term activations: MXFP4 experts only
    w = _weights()
    w.ex_gate_s = 0x10010           # 16- but not 32-byte aligned
    assert _create(lib, _cfg(), w)[0] == b.LMOE_ERR_INVALID_ARG


def test_valid_config_without_gpu_reports_cuda(lib):
    import torch
    from latent_mixture_experts_gb300 import binding as b
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _create(lib, _cfg(), _weights())
    assert st == b.LMOE_ERR_CUDA and not h.value


def test_null_handle_calls(lib):
    from latent_mixture_experts_gb300 import binding as b
    assert lib.lmoe_forward(None, None, 0, None, None, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_route(None, None, 1, None, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_dispatch(None, None, 1, None, None, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_sync_status(None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_destroy(None) == b.LMOE_OK
    assert lib.lmoe_last_launch_count(None) == 0
    assert lib.lmoe_keep_f32_output(None, 1) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_selftest_timeout(None, 5000, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_ep_dispatch(None, None, 1, None, None, None, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_ep_experts(None, None, None, 1, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_ep_combine(None, None, 1, None, None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_qb_update(None, None, 1, None, None, None) == b.LMOE_ERR_INVALID_ARG


def test_tc_peak_rejects_bad_arguments(lib):
    from latent_mixture_experts_gb300 import binding as b
    ms, fl = ctypes.c_float(), ctypes.c_double()
    assert lib.lmoe_tc_peak(9, 10, ctypes.byref(ms), ctypes.byref(fl), None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_tc_peak(0, 0, ctypes.byref(ms), ctypes.byref(fl), None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_tc_peak(0, (1 << 20) + 1, ctypes.byref(ms), ctypes.byref(fl), None) == b.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_tc_peak(0, 10, None, ctypes.byref(fl), None) == b.LMOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    from latent_mixture_experts_gb300 import binding
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            binding.load_library(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved
