"""The in-tree build is content-addressed (CPU): the library is rebuilt when a source,
a flag or the compiler changes, and not because a file's modification time moved."""
import os

import pytest

from paged_kv_cache_87_gb300 import build


@pytest.fixture
def fake_tree(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    lib = tmp_path / "libpagedkv.so"
    lib.write_bytes(b"not a real library")
    monkeypatch.setattr(build, "_inputs", lambda: [str(src)])
    monkeypatch.setattr(build, "LIB", str(lib))
    monkeypatch.setattr(build, "STAMP", str(tmp_path / "libpagedkv.sha256"))
    monkeypatch.setattr(build, "nvcc", lambda: "nvcc")
    monkeypatch.setattr(build, "_nvcc_version", {"nvcc": "Cuda compilation tools, V13.0.88"})
    (tmp_path / "libpagedkv.sha256").write_text(build.digest() + "\n")
    return src


def test_stamp_matches_means_up_to_date(fake_tree):
    assert build.up_to_date()


def test_a_changed_flag_forces_a_rebuild(fake_tree, monkeypatch):
    monkeypatch.setattr(build, "NVCC_FLAGS", build.NVCC_FLAGS + ["-DPKV_SOMETHING=1"])
    assert not build.up_to_date()


def test_extra_flags_and_link_flags_enter_the_digest(fake_tree, monkeypatch):
    assert not build.up_to_date(["-Xptxas", "-v"])
    monkeypatch.setattr(build, "LINK_FLAGS", build.LINK_FLAGS + ["-lcuda"])
    assert not build.up_to_date()


def test_a_changed_compiler_forces_a_rebuild(fake_tree, monkeypatch):
    monkeypatch.setattr(build, "_nvcc_version", {"nvcc": "Cuda compilation tools, V13.1.0"})
    assert not build.up_to_date()


def test_a_changed_source_forces_a_rebuild(fake_tree):
    fake_tree.write_text("__global__ void k() { }\n")
    assert not build.up_to_date()


def test_a_touched_but_unchanged_source_does_not(fake_tree):
    st = os.stat(fake_tree)
    os.utime(fake_tree, (st.st_atime + 3600, st.st_mtime + 3600))
    assert build.up_to_date()


def test_missing_stamp_or_library_forces_a_rebuild(fake_tree):
    os.remove(build.STAMP)
    assert not build.up_to_date()


def test_oracle_build_is_content_addressed(tmp_path, monkeypatch):
    import oracle
    d0 = oracle._digest()
    monkeypatch.setattr(oracle, "_CFLAGS", oracle._CFLAGS + ["-DX=1"])
    assert oracle._digest() != d0
