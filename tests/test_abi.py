"""The C-ABI library builds, loads and exports every symbol include/smp.h
declares; host-side validation answers without touching a GPU."""

import ctypes
import os
import re

import pytest

from spec_verify_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for path in HEADERS:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(smp_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(binding.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_version_and_strings(lib):
    assert lib.smp_abi_version() == 3
    for code in range(6):
        assert lib.smp_status_string(code).decode().startswith(binding.STATUS_NAMES[code])


def test_host_validation_without_gpu(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    # NULL logits, bad sizes and an unknown dtype return before any CUDA call.
    assert lib.smp_sample(null, 4, 8, 0, fake, 0, 0, fake, null, null, null) == 1
    assert lib.smp_sample(fake, 0, 8, 0, fake, 0, 0, fake, null, null, null) == 1
    assert lib.smp_sample(fake, 4, -1, 0, fake, 0, 0, fake, null, null, null) == 1
    assert lib.smp_sample(fake, 4, 8, 7, fake, 0, 0, fake, null, null, null) == 2
    assert lib.smp_sample(fake, 4, (1 << 19) + 1, 0, fake, 0, 0, fake, null, null, null) == 4
    assert lib.smp_sample(ctypes.c_void_p(0x1001), 4, 8, 1, fake, 0, 0, fake, null, null, null) == 1
    assert lib.smp_filter_debug(fake, 4, 8, 0, fake, 0, 0, fake, null, null, null, null, null) == 1
    # pre-pass sampling: history length out of range, history missing, misaligned mask
    assert lib.smp_sample_processed(fake, 4, 8, 0, fake, null, fake, 65, null, 0, 0, fake, null, null, null) == 1
    assert lib.smp_sample_processed(fake, 4, 8, 0, fake, null, null, 4, null, 0, 0, fake, null, null, null) == 1
    assert lib.smp_sample_processed(fake, 4, 8, 0, fake, ctypes.c_void_p(0x1002), null, 0, null, 0, 0, fake,
                                    null, null, null) == 1
    assert lib.smp_sample_processed(fake, 4, 8, 5, fake, null, null, 0, null, 0, 0, fake, null, null, null) == 2
    # a part of a larger batch: the same checks as the pre-pass entry
    assert lib.smp_sample_rows(null, 4, 8, 0, fake, null, null, 0, null, 0, 0, 64, fake, null, null, null) == 1
    assert lib.smp_sample_rows(fake, 4, 8, 0, fake, null, fake, 65, null, 0, 0, 64, fake, null, null, null) == 1
    assert lib.smp_sample_rows(fake, 4, 8, 6, fake, null, null, 0, null, 0, 0, 64, fake, null, null, null) == 2
    assert lib.smp_sample_rows(fake, 4, 8, 0, fake, null, null, 0, null, 0, 0, 64, fake,
                               ctypes.c_void_p(0x1002), null, null) == 1
    assert lib.smp_beam_topk_workspace_bytes(2, 4, 4) == 2 * 4 * 16 * (24 + 4 * 8)   # 16 slices at most
    assert lib.smp_beam_topk_workspace_bytes(2, 33, 4) == 0
    assert lib.smp_beam_topk_workspace_bytes(2, 4, 0) == 0
    assert lib.smp_beam_topk(null, fake, 2, 4, 100, 4, 0, fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.smp_beam_topk(fake, fake, 2, 4, 100, 33, 0, fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.smp_beam_topk(fake, fake, 2, 4, 100, 4, 2, fake, fake, fake, null, fake, 1 << 20, null) == 2
    assert lib.smp_beam_topk(fake, fake, 2, 4, 100, 4, 0, fake, fake, fake, null, null, 1 << 20, null) == 5
    assert lib.smp_beam_topk(fake, fake, 2, 4, 100, 4, 0, fake, fake, fake, null, fake, 10, null) == 5
    assert lib.smp_logit_prepass(null, 4, 8, 0, null, null, 0, null, null, null) == 1
    assert lib.smp_logit_prepass(fake, 4, 8, 0, null, fake, 65, null, null, null) == 1
    assert lib.smp_logit_prepass(fake, 4, 8, 3, null, null, 0, null, null, null) == 2
    assert lib.smp_logit_prepass(ctypes.c_void_p(0x1001), 4, 8, 1, null, null, 0, null, null, null) == 1
    # verify: K out of range, workspace missing or too small
    assert lib.smp_spec_verify(fake, fake, fake, 2, 0, 8, 0, 0, 0, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.smp_spec_verify(fake, fake, fake, 2, 17, 8, 0, 0, 0, fake, fake, null, fake, 1 << 20, null) == 1
    assert lib.smp_spec_verify(fake, fake, fake, 2, 4, 8, 0, 0, 0, fake, fake, null, null, 1 << 20, null) == 5
    need = lib.smp_spec_verify_workspace_bytes(2, 4)
    assert need == 2 * 9 * 32
    assert lib.smp_spec_verify(fake, fake, fake, 2, 4, 8, 0, 0, 0, fake, fake, null, fake, need - 1, null) == 5
    # the per-row-knob entry: the same checks, and a misaligned params pointer
    assert lib.smp_spec_verify_params(fake, fake, fake, 2, 0, 8, 0, fake, 0, 0, fake, fake, null, null, fake,
                                      1 << 20, null) == 1
    assert lib.smp_spec_verify_params(fake, fake, fake, 2, 4, 8, 0, ctypes.c_void_p(0x1002), 0, 0, fake, fake,
                                      null, null, fake, 1 << 20, null) == 1
    assert lib.smp_spec_verify_params(fake, fake, fake, 2, 4, 8, 0, fake, 0, 0, fake, fake,
                                      ctypes.c_void_p(0x1001), null, fake, 1 << 20, null) == 1
    assert lib.smp_spec_verify_params(fake, fake, fake, 2, 4, 8, 9, fake, 0, 0, fake, fake, null, null, fake,
                                      1 << 20, null) == 2
    assert lib.smp_spec_verify_params(fake, fake, fake, 2, 4, 8, 0, null, 0, 0, fake, fake, null, null, null,
                                      1 << 20, null) == 5
    assert lib.smp_spec_verify_rows(fake, fake, fake, 2, 17, 8, 0, null, 0, 0, 32, fake, fake, null, null, fake,
                                    1 << 20, null) == 1
    assert lib.smp_spec_verify_rows(fake, fake, fake, 2, 4, 8, 0, null, 0, 0, 32, fake, fake, null, null, null,
                                    1 << 20, null) == 5
    assert lib.smp_spec_verify_workspace_bytes(0, 4) == 0
    assert lib.smp_spec_verify_workspace_bytes(2, 17) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(binding.SmpError):
        binding.load()
