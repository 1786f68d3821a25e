"""The binding has no CPU fallback: without the built library (and without a
way to build it) every entry point raises instead of computing anything."""
import pytest

import sparse_decode_attention_gb300 as kvr
from sparse_decode_attention_gb300 import _build


@pytest.fixture
def no_library(tmp_path, monkeypatch):
    monkeypatch.setattr(kvr, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libkvr.so"))
    yield


def test_load_refuses_a_missing_library(no_library):
    with pytest.raises(RuntimeError, match="not built"):
        kvr.load(build_if_missing=False)


def test_build_without_nvcc_raises(no_library, monkeypatch):
    monkeypatch.setattr(_build.shutil, "which", lambda name: None)
    monkeypatch.setattr(_build.os.path, "exists",
                        lambda p: False if p.endswith("nvcc") or p == _build.LIB else True)
    with pytest.raises(RuntimeError, match="nvcc not found"):
        kvr.load()


def test_entry_points_go_through_the_library(no_library, monkeypatch):
    monkeypatch.setattr(_build.shutil, "which", lambda name: None)
    monkeypatch.setattr(_build.os.path, "exists",
                        lambda p: False if p.endswith("nvcc") or p == _build.LIB else True)
    shape = kvr.Shape(1, 4, 4, 64, 128, "f32")
    with pytest.raises(RuntimeError):
        kvr.kvr_status_string(0)
    with pytest.raises(RuntimeError):
        kvr.kvr_codes_bytes(shape)
