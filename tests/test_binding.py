"""The Python binding refuses arguments the library cannot take, before any
call reaches the device (CPU only: CPU tensors stand in for wrong devices)."""
import pytest

from rank_orthonormalized_optimizer_03_b300 import dion


def cpu_mat(m=64, n=32, r=8, **kw):
    import torch
    d = dict(X=torch.zeros(m, n), G=torch.zeros(m, n, dtype=torch.bfloat16), R=torch.zeros(m, n),
             V=torch.zeros(n, r), eta=0.01, beta=0.95, variant="orth")
    d.update(kw)
    return d


def test_plan_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensor"):
        dion.Plan([cpu_mat()])


def test_plan_refuses_an_empty_batch():
    with pytest.raises(ValueError, match="at least one"):
        dion.Plan([])


@pytest.mark.parametrize("bad, match", [
    (dict(variant="muon"), "variant"),
    (dict(V=None), "V must"),
    (dict(R=None), "R must"),
])
def test_descriptor_checks(bad, match):
    import torch
    d = cpu_mat()
    if "V" in bad:
        d["V"] = torch.zeros(32, 8)[:, :4]          # not contiguous
    elif "R" in bad:
        d["R"] = torch.zeros(64, 32).t()            # wrong shape / strides
    else:
        d.update(bad)
    with pytest.raises(ValueError, match=match):
        dion.make_desc(d["X"], d["G"], d["R"], d["V"], d["eta"], d["beta"], d["variant"])


def test_orth_noalloc_refuses_host_tensors():
    import torch
    with pytest.raises(ValueError, match="CUDA tensor"):
        dion.orth_noalloc(torch.zeros(128, 8), torch.zeros(128, 8))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libdion.so there is no fallback: every entry point raises."""
    monkeypatch.setattr(dion, "LIB_PATH", str(tmp_path / "libdion.so"))
    monkeypatch.setattr(dion, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        dion.lib()
    with pytest.raises(RuntimeError, match="not built"):
        dion.Plan([cpu_mat()])
    with pytest.raises(RuntimeError, match="not built"):
        dion.MuonPlan([dict(X=None, G=None, B=None, eta=0.01, mu=0.9)])
