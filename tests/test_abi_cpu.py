"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports
every function include/spin.h declares, and rejects bad configurations before touching
the device."""
import ctypes
import subprocess

import pytest

from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn


def test_exports_every_declared_symbol(spin_lib):
    names = spin.header_functions()
    assert len(names) >= 9
    L = spin.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", spin.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_version(spin_lib):
    assert spin.version().startswith("spin-gb300") and "sm_103a" in spin.version()


def test_workspace_size(spin_lib):
    cfg = spin.make_config(**syn.CONFIGS["serving"].config_fields())
    ws = spin.workspace_size(cfg, 1)
    assert ws >= 4 * 96 * cfg.max_blocks and ws % 256 == 0
    assert spin.workspace_size(cfg, 4) >= 4 * ws - 256 if cfg.max_rows >= 4 else True


@pytest.mark.parametrize("field,value,code", [
    ("block", 32, 1), ("n_req", 0, 1), ("max_rows", 9, 1), ("kv_heads", 3, 2),
    ("q_dtype", 2, 4), ("k_dtype", 7, 4), ("top_k", 0, 1), ("rho_bp", 10001, 1),
    ("gamma_bp", -1, 1), ("alpha", 1.5, 1), ("combine", 2, 1), ("score_path", 9, 1),
    ("max_slots", 0, 3), ("pooling", 5, 1), ("explore", 2, 1), ("reserved", 1, 1),
])
def test_config_validation(spin_lib, field, value, code):
    fields = syn.CONFIGS["pr1"].config_fields()
    cfg = spin.make_config(**fields)
    setattr(cfg, field, value)
    size = ctypes.c_size_t(0)
    rc = spin.lib().spin_workspace_size(ctypes.byref(cfg), 1, ctypes.byref(size))
    assert rc == code
    assert spin.lib().spin_last_error_string().decode() != ""
    # every entry point validates the configuration first (no device access happens)
    rc = spin.lib().spin_select_blocks(ctypes.byref(cfg), None, None, None, None, None, None, 1,
                                       None, 0, 0, None, None, None, None, None, 0, None, None)
    assert rc == code


def test_null_pointers_rejected(spin_lib):
    cfg = spin.make_config(**syn.CONFIGS["pr1"].config_fields())
    L = spin.lib()
    assert L.spin_topk(ctypes.byref(cfg), None, None, None, None, 1, None, None, None) == 1
    assert L.spin_update_ema(ctypes.byref(cfg), *([None] * 11)) == 1
    assert L.spin_commit_mtp(ctypes.byref(cfg), None, None, None, None, None, 1, *([None] * 7)) == 1
    assert L.spin_indexer_score(ctypes.byref(cfg), None, None, None, None, 0, None, 0, None, None,
                                None, 1, None, None, None) == 1
    # rows beyond max_rows
    assert L.spin_topk(ctypes.byref(cfg), None, None, None, None, 2, None, None, None) == 2
    # the device-step selection needs its step pointer
    assert L.spin_select_blocks_dstep(ctypes.byref(cfg), *([None] * 6), 1, None, None, 0,
                                      *([None] * 5), 0, None, None) == 1
    assert "step_dev" in L.spin_last_error_string().decode()


def test_library_refuses_to_run_without_build(tmp_path, monkeypatch):
    """No silent fallback: a missing library raises."""
    monkeypatch.setattr(spin, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(spin, "_LIB", None)
    with pytest.raises(RuntimeError):
        spin.lib()


def test_config_struct_layout(tmp_path):
    """The binding's spin_config has the C struct's size and field offsets (gcc on the
    header, no GPU)."""
    import os
    names = [f[0] for f in spin.SpinConfig._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "spin.h"\nint main(void) {\n'
                   '    printf("%zu", sizeof(spin_config));\n' +
                   "".join('    printf(" %%zu", offsetof(spin_config, %s));\n' % n for n in names) +
                   "    return 0;\n}\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(spin.HEADER))
    subprocess.run(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(spin.SpinConfig)
    assert vals[1:] == [getattr(spin.SpinConfig, n).offset for n in names]


def test_ablation_modes_refused_on_the_host(spin_lib):
    """The one-row ablations (A2 block states, block-age exploration) and the age entry points
    are refused before any device access: every pointer the checks read first is NULL, so a
    missing check would end at the NULL-pointer check, never at a launch."""
    L = spin.lib()
    fake_age = ctypes.c_void_p(256)
    err = lambda: L.spin_last_error_string().decode()

    def cfg_of(**kw):
        return spin.make_config(**syn.CONFIGS["pr1"].replace(rows=2, mean_accept=1.5, **kw).config_fields())

    a2 = cfg_of(pooling="a2")
    assert L.spin_select_blocks(ctypes.byref(a2), *([None] * 6), 2, None, 0, 0, *([None] * 5), 0, None,
                                None) == 4 and "A2" in err()
    assert L.spin_commit_mtp(ctypes.byref(a2), *([None] * 5), 2, *([None] * 7)) == 4 and "A2" in err()
    assert L.spin_select_blocks_noalloc(ctypes.byref(a2), *([None] * 6), 2, None, 0, 0,
                                        *([None] * 6)) == 4 and "A2" in err()

    age = cfg_of(explore="age")
    assert L.spin_select_blocks(ctypes.byref(age), *([None] * 6), 1, None, 0, 0, *([None] * 5), 0, None,
                                None) == 1 and "spin_select_blocks_age" in err()
    assert L.spin_select_blocks_noalloc(ctypes.byref(age), *([None] * 6), 1, None, 0, 0,
                                        *([None] * 6)) == 1 and "spin_select_blocks_age" in err()
    assert L.spin_select_blocks_age(ctypes.byref(age), *([None] * 6), 2, None, 0, 0, fake_age, *([None] * 5), 0,
                                    None, None) == 4 and "one query row" in err()
    assert L.spin_select_blocks_age(ctypes.byref(age), *([None] * 6), 1, None, 0, 0, None, *([None] * 5), 0,
                                    None, None) == 1 and "block_age is NULL" in err()
    assert L.spin_update_ema_age(ctypes.byref(age), *([None] * 9), None, 0, None, None) == 1 \
        and "block_age is NULL" in err()

    plain = cfg_of()
    assert L.spin_select_blocks_age(ctypes.byref(plain), *([None] * 6), 1, None, 0, 0, fake_age,
                                    *([None] * 5), 0, None, None) == 1 and "SPIN_EXPLORE_BLOCK_AGE" in err()
    # the stacked selection has no age array: refused under BLOCK_AGE before any pointer check
    assert L.spin_select_blocks_layers(ctypes.byref(age), 2, 0, *([None] * 6), 1, None, 0, None,
                                       *([None] * 5), 0, None, None) == 1 and "spin_select_blocks_age" in err()
