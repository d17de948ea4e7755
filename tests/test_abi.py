"""The C-ABI library builds, loads, and exports every symbol include/dflash.h declares
(no compute calls: these run without a GPU)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]*?\b(dflash\w*)\s*\(", src)))


def test_header_declares_the_step_calls():
    names = declared()
    for n in ("dflash_ctx_project", "dflash_draft_block", "dflash_lm_head_topk", "dflash_accept",
              "dflash2_conv", "dflash2_select", "dflash_create", "dflash_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from block_diffusion_speculative_project_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    for n in declared():
        assert hasattr(lib, n), f"{n} declared in dflash.h but not exported"


def test_binding_wraps_every_symbol_and_validates_without_gpu():
    from block_diffusion_speculative_project_gb300 import dflash
    assert set(dflash.EXPORTED) == set(declared())
    cfg = dflash.dflash_config(D=256, Dt=256, L=5, N=2, Hq=4, Hkv=4, hd=96, F=688, V=4096, B=8,
                               k_top=16, rope_base=1e4, eps=1e-6, mask_id=4095, Cmax=80,
                               max_batch=1, max_proj_rows=64, conv_group=16, sel_dim=256)
    try:
        dflash.dflash_create(cfg)
        raise AssertionError("hd=96 must be rejected")
    except dflash.DflashError as e:
        assert e.code == dflash.DFLASH_ERR_UNSUPPORTED_SHAPE


def test_film_relay_config_is_validated_without_gpu():
    from block_diffusion_speculative_project_gb300 import dflash
    base = dict(D=256, Dt=256, L=5, N=2, Hq=4, Hkv=4, hd=64, F=688, V=4096, B=8, k_top=16,
                rope_base=1e4, eps=1e-6, mask_id=4095, Cmax=80, max_batch=1, max_proj_rows=64,
                conv_group=16, sel_dim=256)
    for flags, film_dim, code in ((dflash.FLAG_FILM, 64, dflash.DFLASH_ERR_INVALID_ARG),
                                  (dflash.FLAG_FILM | dflash.FLAG_RELAY, 96,
                                   dflash.DFLASH_ERR_UNSUPPORTED_SHAPE),
                                  (dflash.FLAG_FILM | dflash.FLAG_RELAY, 0,
                                   dflash.DFLASH_ERR_UNSUPPORTED_SHAPE)):
        cfg = dflash.dflash_config(flags=flags, film_dim=film_dim, **base)
        try:
            dflash.dflash_create(cfg)
            raise AssertionError(f"flags={flags} film_dim={film_dim} must be rejected")
        except dflash.DflashError as e:
            assert e.code == code, (flags, film_dim, e)


def test_paged_config_is_validated_without_gpu():
    from block_diffusion_speculative_project_gb300 import dflash
    base = dict(D=256, Dt=256, L=5, N=2, Hq=4, Hkv=4, hd=64, F=688, V=4096, B=8, k_top=16,
                rope_base=1e4, eps=1e-6, mask_id=4095, max_batch=1, max_proj_rows=64,
                conv_group=16, sel_dim=256)
    for Cmax, num_pages, code in ((80, 4, dflash.DFLASH_ERR_UNSUPPORTED_SHAPE),   # Cmax % 64
                                  (128, -1, dflash.DFLASH_ERR_INVALID_ARG),
                                  (128, 1 << 30, dflash.DFLASH_ERR_UNSUPPORTED_SHAPE)):  # rows >= 2^31
        cfg = dflash.dflash_config(Cmax=Cmax, num_pages=num_pages, **base)
        try:
            dflash.dflash_create(cfg)
            raise AssertionError(f"Cmax={Cmax} num_pages={num_pages} must be rejected")
        except dflash.DflashError as e:
            assert e.code == code, (Cmax, num_pages, e)
    try:
        dflash.dflash_set_block_table(None, None)
        raise AssertionError("a NULL handle must be rejected")
    except dflash.DflashError as e:
        assert e.code == dflash.DFLASH_ERR_INVALID_ARG


def test_seeded_block_tables_are_permutations():
    import numpy as np
    import dflash_inputs as di
    t = di.block_table(5, 4 * di.PAGE_ROWS, seed=3)
    assert t.shape == (5, 4) and t.dtype == np.int32
    assert sorted(t.ravel().tolist()) == list(range(20))
    assert np.array_equal(t, di.block_table(5, 4 * di.PAGE_ROWS, seed=3))
    assert not np.array_equal(t, di.block_table(5, 4 * di.PAGE_ROWS, seed=4))
