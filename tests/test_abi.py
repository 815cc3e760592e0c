"""C-ABI checks that need no GPU: the library builds and loads, every symbol the
header declares is exported, host-side arithmetic matches the oracle bit for bit,
and argument errors come back as status codes."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import sched

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qi():
    import diffusion_transformer_text_gb300 as q
    q.build()
    q.lib()
    return q


def _declared():
    with open(os.path.join(ROOT, "include", "qidit.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qi_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(qi):
    names = _declared()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", qi.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (qi_[a-z0-9_]+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(qi.SYMBOLS) == set(names)


def test_library_has_sm103a_code(qi):
    out = subprocess.run(["cuobjdump", "--list-elf", qi.LIB], capture_output=True, text=True).stdout
    assert "sm_103a" in out


@pytest.mark.parametrize("N", [64, 256, 576, 1024, 4096, 16384])
@pytest.mark.parametrize("steps", [2, 3, 25, 40])
def test_flow_sigmas_bit_exact(qi, N, steps):
    s, t = qi.flow_sigmas(steps, N)
    rs, rt = sched.flow_sigmas(steps, N)
    assert s.tobytes() == rs.tobytes()
    assert t.tobytes() == rt.tobytes()


def test_single_step_is_rejected(qi):
    """One step: the only sigma is 1, so the terminal stretch is 0/0 (the oracle gives NaN)."""
    with np.errstate(invalid="ignore"):
        rs, _ = sched.flow_sigmas(1, 256)
    assert np.isnan(rs[0])
    with pytest.raises(qi.QiError) as e:
        qi.flow_sigmas(1, 256)
    assert e.value.status == 2


def test_flow_sigmas_custom_constants(qi):
    p = dict(base_shift=0.3, max_shift=1.1, base_seq=128, max_seq=4096, shift_terminal=0.05, train_steps=1000)
    s, t = qi.flow_sigmas(30, 2000, p)
    rs, rt = sched.flow_sigmas(30, 2000, 0.3, 1.1, 128, 4096, 0.05, 1000)
    assert s.tobytes() == rs.tobytes() and t.tobytes() == rt.tobytes()


def test_kv_cache_bytes(qi):
    assert qi.kv_cache_bytes(32, 494) == 2 * 32 * 494 * 4096 * 2
    assert qi.kv_cache_bytes(0, 5) == 0


def test_status_codes(qi):
    L = qi.lib()
    sig = np.zeros(41, np.float32)
    ts = np.zeros(40, np.float32)
    assert L.qi_flow_sigmas(0, 256, None, sig.ctypes.data, ts.ctypes.data) == 2       # SHAPE
    assert L.qi_flow_sigmas(40, 256, None, None, ts.ctypes.data) == 1                # INVALID_ARG
    assert b"NULL" in L.qi_last_error()
    h = ctypes.c_void_p()
    bad = qi.DitConfig(0, 8, 64)
    assert L.qi_dit_create(ctypes.byref(bad), 0, ctypes.byref(h)) == 2
    bad = qi.DitConfig(1, 8, 16385)
    assert L.qi_dit_create(ctypes.byref(bad), 0, ctypes.byref(h)) == 2
    assert L.qi_dit_create(None, 0, ctypes.byref(h)) == 1
    assert L.qi_dit_destroy(None) == 0
    assert L.qi_rope_tables(0, 8, 8, 10000.0, None, None, None, None, None) == 2
    assert L.qi_rope_tables(8, 8, 8, 0.5, None, None, None, None, None) == 1
    assert L.qi_pack_noise(None, 8, 8, None, None) == 1
    assert L.qi_euler_update(None, None, 8, 1.0, 0.5, None) == 1
    assert L.qi_dit_step(None, None, 8, None, 8, 0.5, None, None, None, None, None, 0, None) == 1
    assert L.qi_attention_f16(None, None, None, None, 1, 0, 1, 1, None) == 1
    assert L.qi_gemv_bf16(None, 4096, None, None, 16, None, 0, None) == 1
    assert L.qi_dit_profile(None, 1) == 1
    assert L.qi_dit_profile_classes(None, 8, 1) == 1


def test_kv_slots_range(qi):
    L = qi.lib()
    h = ctypes.c_void_p()
    assert L.qi_dit_create(ctypes.byref(qi.DitConfig(1, 8, 64, 3)), 0, ctypes.byref(h)) == 2
    assert L.qi_dit_create(ctypes.byref(qi.DitConfig(1, 8, 64, -1)), 0, ctypes.byref(h)) == 2
    assert L.qi_dit_step_cfg(None, None, 64, 0.5, 2.0, None, 8, None, None, None, None, None, 8, None, None,
                             None, None, None, 0, None) == 1


@pytest.mark.parametrize("N", [256, 1024, 4096, 16384])
@pytest.mark.parametrize("steps", [2, 3, 20, 40])
def test_dpmpp2m_coeffs_bit_exact(qi, N, steps):
    s, _ = sched.flow_sigmas(steps, N)
    for i in range(steps):
        got = qi.dpmpp2m_coeffs(s, i)
        ref = sched.dpmpp2m_coeffs(s, i)
        assert got[0] == ref[0], (i, got, ref)
        assert np.array(got[1:], np.float32).tobytes() == np.array(ref[1:], np.float32).tobytes(), (i, got, ref)


def test_dpmpp2m_coeffs_custom_schedule_and_errors(qi):
    s = np.array([0.9, 0.6, 0.35, 0.1, 0.0], np.float32)
    for i in range(4):
        got, ref = qi.dpmpp2m_coeffs(s, i), sched.dpmpp2m_coeffs(s, i)
        assert got[0] == ref[0] and np.array(got[1:], np.float32).tobytes() == np.array(ref[1:], np.float32).tobytes()
    with pytest.raises(qi.QiError) as e:
        qi.dpmpp2m_coeffs(s, 4)                    # step index past the end
    assert e.value.status == 1
    with pytest.raises(qi.QiError) as e:
        qi.dpmpp2m_coeffs(np.array([0.5, 0.7, 0.0], np.float32), 0)   # increasing
    assert e.value.status == 1
    with pytest.raises(qi.QiError) as e:
        qi.dpmpp2m_coeffs(np.array([1.5, 0.7, 0.0], np.float32), 1)   # sigma above 1
    assert e.value.status == 1


def test_debug_inject_arguments(qi):
    L = qi.lib()
    assert L.qi_debug_inject(None, 9, 0) == 1           # unknown kind
    assert L.qi_debug_inject(None, 1, 0) == 1           # allocation index must be >= 1
    assert L.qi_debug_inject(None, 2, 0) == 1           # a stall needs a handle
    assert L.qi_debug_inject(None, 0, 0) == 0
