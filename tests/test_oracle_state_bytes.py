"""State-memory pins from the pages and shape pins of the seeded workloads.

* "Fused Optimizers and State Precision", section 05: 100M parameters -> two
  fp32 moments 800 MB, two 16-bit moments 400 MB, two 8-bit codes 200 MB
  (+ low-bit metadata).
* ApexW Unsloth benchmark page (results table): optimizer state 185.501 MB
  (AdamW), 92.751 MB (ApexW Compact), 47.101 MB (ApexW 8bit) for the
  24.3M-parameter LoRA run; the figures are MiB to three decimals.
"""
import numpy as np

import workloads
from oracle import state_bytes


def test_lora_state_memory_matches_benchmark_page():
    wl = workloads.lora()
    assert len(wl.tensors) == 392
    assert wl.total_numel == 24_313_856
    mib = lambda k: round(state_bytes.state_bytes(wl.numels, k) / 2 ** 20, 3)
    assert mib("f32") == 185.501
    assert mib("bf16") == 92.751
    assert mib("int8") == 47.101


def test_100m_payload_matches_section_05():
    n = [100_000_000]
    assert state_bytes.state_bytes(n, "f32", with_step=False) == 800_000_000
    assert state_bytes.state_bytes(n, "bf16", with_step=False) == 400_000_000
    b8 = state_bytes.state_bytes(n, "int8", with_step=False)
    assert b8 - 200_000_000 == 8 * (-(-100_000_000 // 256))   # the metadata


def test_workload_shapes():
    assert workloads.few_large().total_numel == 134_217_728
    ll = workloads.llama3_8b()
    assert len(ll.tensors) == 291 and ll.total_numel == 8_030_261_248
    ms = workloads.many_small()
    assert len(ms.tensors) == 20_050
    assert ms.total_numel == 117_880_217 + 50 * 4096 * 1024
    assert ms.found_inf(5) and not ms.found_inf(4)
    p = ms.present(3)
    assert 0.08 < 1 - p.mean() < 0.12
    assert np.array_equal(p, ms.present(3)) and not np.array_equal(p, ms.present(4))


def test_seeded_fills_are_deterministic():
    import torch
    wl = workloads.tiny()
    a = workloads.init_param(wl, 2)
    b = workloads.init_param(wl, 2)
    assert torch.equal(a, b)
    g1 = workloads.grad(wl, 0, 1)
    assert g1.tolist() == [np.float32(0.1), np.float32(-0.2)]
    assert torch.equal(workloads.grad(wl, 1, 3), workloads.grad(wl, 1, 3))
    assert not torch.equal(workloads.grad(wl, 1, 3), workloads.grad(wl, 1, 4))
    lo = workloads.lora(layers=1)
    g = workloads.grad(lo, 0, 1)
    zb = lo.zero_blocks(0)
    flat = g.view(-1)
    for b in zb:
        assert torch.all(flat[b * 256:(b + 1) * 256] == 0)


def test_selective_fp32_for_small_tensors():
    # 100 and 4095 elements stay fp32 (8 B each), 4096 and 5000 are coded
    # (2 B each plus two fp32 scales per 256-block), plus a 4 B step per tensor
    from oracle.state_bytes import kind_for
    sb = state_bytes.state_bytes
    numels = [100, 5000, 4095, 4096]
    want = (8 * (100 + 4095) + 2 * (5000 + 4096) + 2 * 4 * (20 + 16) + 4 * 4)
    for kind in ("int8", "int8uv", "dyn8"):
        assert sb(numels, kind, min_8bit_size=4096) == want
        assert kind_for(4095, kind, 4096) == "f32" and kind_for(4096, kind, 4096) == kind
    assert kind_for(10, "bf16", 4096) == "bf16"       # only 8-bit kinds are affected
