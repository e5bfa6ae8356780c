"""The C-ABI library builds, loads without a GPU and exports every symbol the
public header declares; host-side validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "fk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fk_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = _declared()
    for n in ("fk_model_create", "fk_forward", "fk_session_prefill", "fk_decode_step", "fk_model_free",
              "fk_gemm_bf16", "fk_sync_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import transformer_decoder_forward_bf16_gb300 as fk
    lib = fk.load()
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.fk_version().decode().startswith("fk ")
