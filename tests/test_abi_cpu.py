"""C ABI checks that need no GPU: the library loads, exports every entry point the header
declares, and rejects invalid configurations on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "dg_sampler.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = set(re.findall(r"\b(dg_[a-z_]+)\s*\(", txt))
    names -= {"dg_resid_fn"}  # a function-pointer type, not an entry point
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("dg_sampler_create", "dg_denoise_step", "dg_run", "dg_destroy", "dg_workspace_size"):
        assert required in names


def test_library_exports_every_declared_symbol():
    import uniform_state_discrete_gb300 as dg
    lib = ctypes.CDLL(dg.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared_functions()) <= set(dg._SIGS)


def test_struct_layouts_match_header_sizes():
    import uniform_state_discrete_gb300 as dg
    assert ctypes.sizeof(dg.dg_config) == 88
    assert ctypes.sizeof(dg.dg_slot) == 56
    assert ctypes.sizeof(dg.dg_state) == 64


@pytest.mark.parametrize("field,value", [("vocab", 1), ("hidden", 100), ("hidden", 0), ("canvas_len", 0),
                                         ("canvas_len", 1025), ("num_inference_steps", 0),
                                         ("num_inference_steps", 1025), ("t_min", 0.0), ("t_max", -1.0),
                                         ("entropy_bound", -0.1), ("confidence", -1.0), ("n_canvases", 0),
                                         ("gen_blocks", 0), ("rms_eps", -1.0), ("max_active", 5),
                                         ("softcap", -1.0), ("softcap", float("inf")), ("stability", 0),
                                         ("stability", 1025)])
def test_invalid_configs_rejected_on_host(field, value):
    import uniform_state_discrete_gb300 as dg
    kw = dict(vocab=2048, hidden=128, canvas_len=16, n_canvases=2)
    cfg = dg.make_config(**kw)
    setattr(cfg, field, value)
    assert dg.dg_workspace_size(cfg) == 0
    h = ctypes.c_void_p()
    st = dg.lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(16), None, ctypes.c_void_p(256), 1 << 30,
                                  None, ctypes.byref(h))
    assert st == dg.DG_ERR_ARG and not h.value
    assert dg.lib.dg_last_error(None)


def test_unsupported_knobs_and_bad_pointers():
    import uniform_state_discrete_gb300 as dg
    h = ctypes.c_void_p()
    # any stability in [1, 1024] is a valid config of the same size
    assert dg.dg_workspace_size(dg.make_config(2048, 128, 16, stability=3)) == \
        dg.dg_workspace_size(dg.make_config(2048, 128, 16)) > 0
    # the two commit modes size the same workspace; any other mode is an invalid config
    cfg = dg.make_config(2048, 128, 16, mode=dg.DG_REACCEPT)
    assert dg.dg_workspace_size(cfg) == dg.dg_workspace_size(dg.make_config(2048, 128, 16)) > 0
    cfg = dg.make_config(2048, 128, 16, mode=2)
    assert dg.dg_workspace_size(cfg) == 0
    assert dg.lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(16), None, ctypes.c_void_p(256), 1 << 30,
                                    None, ctypes.byref(h)) == dg.DG_ERR_ARG
    cfg = dg.make_config(2048, 128, 16)
    need = dg.dg_workspace_size(cfg)
    assert need > 0
    assert dg.lib.dg_sampler_create(ctypes.byref(cfg), None, None, ctypes.c_void_p(256), need, None,
                                    ctypes.byref(h)) == dg.DG_ERR_ARG
    assert dg.lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(24), None, ctypes.c_void_p(256), need, None,
                                    ctypes.byref(h)) == dg.DG_ERR_ALIGN
    assert dg.lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(16), None, ctypes.c_void_p(256), need - 1,
                                    None, ctypes.byref(h)) == dg.DG_ERR_WORKSPACE
    assert dg.lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(16), None, ctypes.c_void_p(128), need, None,
                                    ctypes.byref(h)) == dg.DG_ERR_ALIGN
    seeds_ok = dg.make_config(2048, 128, 16, n_canvases=2, admit_tick=[0, -1])
    assert dg.dg_workspace_size(seeds_ok) == 0
    for st in range(9):
        assert dg.lib.dg_status_string(st).startswith(b"DG_")
    dg.lib.dg_destroy(None)  # NULL-safe


def test_workspace_grows_with_batch_and_model():
    import uniform_state_discrete_gb300 as dg
    small = dg.dg_workspace_size(dg.make_config(32768, 1024, 256))
    big = dg.dg_workspace_size(dg.make_config(262144, 2816, 256, n_canvases=16))
    assert 0 < small < big
    assert small % 256 == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """No CPU fallback: a missing shared library is an import error."""
    import importlib.util
    src = os.path.join(ROOT, "uniform_state_discrete_gb300", "__init__.py")
    pkg = tmp_path / "uniform_state_discrete_gb300"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("dg_copy", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_vocab_split_rules():
    """Vocabulary-parallel configs: the rank must lie in [0, vocab_ranks) and there can be no more
    ranks than vocabulary chunks; dg_vocab_slice cuts V into contiguous, tile-aligned slices."""
    import uniform_state_discrete_gb300 as dg
    for ranks, rank, ok in ((2, 0, True), (2, 1, True), (2, 2, False), (3, -1, False), (9, 0, False), (8, 7, True)):
        cfg = dg.make_config(2048, 128, 16, vocab_ranks=ranks, vocab_rank=rank)  # 8 tiles -> 8 chunks
        assert (dg.dg_workspace_size(cfg) > 0) == ok, (ranks, rank)
    for V in (2048, 1000, 262144, 300000):
        for G in (1, 2, 3, 4, 7):
            if G > -(-V // 256):
                continue  # more ranks than chunks
            cuts = [dg.vocab_slice(V, G, r) for r in range(G)]
            assert cuts[0][0] == 0 and cuts[-1][1] == V
            assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:]))
            assert all(c[0] % 256 == 0 and c[1] > c[0] for c in cuts)
    with pytest.raises(dg.DGError):
        dg.vocab_slice(1000, 5, 0)  # 4 tiles, 4 chunks


def test_release_build_has_no_debug_checks():
    """dg_debug_check answers DG_ERR_UNSUPPORTED in the release build (no guards, no index checks) and
    DG_ERR_ARG for a NULL sampler."""
    import uniform_state_discrete_gb300 as dg
    assert dg.lib.dg_debug_check(None, None) == dg.DG_ERR_ARG
    assert dg.lib.dg_status_string(dg.DG_ERR_BOUNDS) == b"DG_ERR_BOUNDS"
