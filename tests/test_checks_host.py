"""Host side of the checks build (CPU only): guard bands around allocated
buffers report writes outside a buffer and nothing else; the library declares
and exports moe_checks_read."""
import torch

import moe_expert_layer_softmax_gb300 as m


def test_guard_bands_catch_writes_past_either_end(monkeypatch):
    monkeypatch.setattr(m, "CHECKS", True)
    monkeypatch.setattr(m, "_guarded", {})
    a = m._alloc((100, 3), torch.int32, "cpu")
    b = m._alloc((4096,), torch.uint8, "cpu", zero=True)
    assert a.shape == (100, 3) and a.dtype == torch.int32
    assert int(b.sum()) == 0
    a.fill_(7)                          # in bounds: no report
    b.fill_(255)
    assert m.check_canaries() == []
    base_a = a.view(-1).view(torch.uint8)
    # one byte past the end of `a`, one byte before the start of `b`
    torch.as_strided(base_a, (1,), (1,), base_a.storage_offset() + base_a.numel()).fill_(0)
    torch.as_strided(b, (1,), (1,), b.storage_offset() - 1).fill_(0)
    bad = m.check_canaries()
    assert len(bad) == 2
    assert any("back guard" in x for x in bad) and any("front guard" in x for x in bad)
    del a
    assert len(m.check_canaries()) == 1      # a freed buffer is no longer checked


def test_normal_mode_allocates_plain_tensors(monkeypatch):
    monkeypatch.setattr(m, "CHECKS", False)
    t = m._alloc((8, 8), torch.float32, "cpu", zero=True)
    assert t.is_contiguous() and t.storage_offset() == 0 and float(t.abs().sum()) == 0.0


def test_checks_read_is_exported():
    assert "moe_checks_read" in m.EXPORTS
    with open(m.os.path.join(m._PKG, "..", "include", "moe.h")) as fh:
        assert "moe_checks_read(int32_t* flags, int32_t reset)" in fh.read()
