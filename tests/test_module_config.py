"""Host-side checks of SparseLandmarkAttention's configuration (no GPU)."""
import pytest


def test_window_and_globals_from_environment(monkeypatch):
    from long_context_sparse_landmark_gb300 import SparseLandmarkAttention
    monkeypatch.setenv("SPARSE_WINDOW", "1024")
    monkeypatch.setenv("SPARSE_GLOBAL_TOKENS", "64")
    m = SparseLandmarkAttention()
    assert (m.window, m.num_global) == (1024, 64)
    m = SparseLandmarkAttention(window=7, num_global=0)
    assert (m.window, m.num_global) == (7, 0)


def test_defaults_without_environment(monkeypatch):
    from long_context_sparse_landmark_gb300 import SparseLandmarkAttention
    monkeypatch.delenv("SPARSE_WINDOW", raising=False)
    monkeypatch.delenv("SPARSE_GLOBAL_TOKENS", raising=False)
    m = SparseLandmarkAttention()
    assert (m.window, m.num_global) == (4096, 512)


def test_bad_configuration_rejected():
    from long_context_sparse_landmark_gb300 import SparseLandmarkAttention
    with pytest.raises(ValueError):
        SparseLandmarkAttention(window=0)
