"""GPU parity of the 8-bit state variants against the oracle, through the C ABI.

CS_STATE_INT8_UV (unsigned linear v codec), CS_STATE_DYN8 (dynamic-exponent
codebook) and selective fp32 moments for small tensors in an 8-bit plan:
oracle-forced steps over ragged tensors spanning several work units for
fp32 / bf16 / fp16 params, misaligned buffers (the scalar path), the step
contract (grad=None, found_inf) with snapshots, fp32 master weights with the
codebook, and full-size workloads on sampled 256-element blocks. Codes must
agree within one position of their codebook and scales within 1e-6; almost
all codes must agree exactly.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.parity_harness import Harness, check_bars, code_index

pytestmark = pytest.mark.gpu

RAGGED = [1, 3, 4, 5, 255, 256, 257, 1000, 4099, 70001]
VARIANTS = ["int8uv", "dyn8"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def _exact_code_fraction(h):
    same = total = 0
    for i, o in enumerate(h.ostates):
        if o.state_kind == "f32":
            continue
        _, m, v, _, _ = h._gpu_state(i)
        for g, r, which in ((m, o.m, "m"), (v, o.v, "v")):
            same += int(np.sum(code_index(g, o.state_kind, which) ==
                               code_index(r, o.state_kind, which)))
            total += g.size
    return same / max(total, 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", VARIANTS)
def test_variant_forced_ragged(kind, dtype):
    wl = workloads.mixed(RAGGED, param_dtype=dtype, groups=2, steps=6)
    h = Harness(wl, kind, unit_elems=1024)
    res = h.run(forced=True)
    check_bars(res, kind, dtype, forced=True)
    assert _exact_code_fraction(h) > 0.999


@pytest.mark.parametrize("kind", VARIANTS)
def test_variant_misaligned_buffers(kind):
    wl = workloads.mixed([5, 257, 4099], param_dtype="bf16", steps=4)
    h = Harness(wl, kind, misalign=True)
    res = h.run(forced=True)
    check_bars(res, kind, "bf16", forced=True)


@pytest.mark.parametrize("kind", VARIANTS)
def test_variant_contract_none_and_found_inf(kind):
    wl = workloads.mixed([300, 5000, 70001], steps=8, none_fraction=0.3, found_inf_steps=(3,),
                         grad_prescale=1024.0)
    h = Harness(wl, kind)
    res = h.run(forced=True)      # snapshots are checked on None tensors and skipped steps
    check_bars(res, kind, "f32", forced=True)


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
def test_selective_fp32_small_tensors(kind):
    sizes = [1, 100, 255, 4095, 4096, 5000, 70001]
    wl = workloads.mixed(sizes, param_dtype="bf16", groups=2, steps=6)
    h = Harness(wl, kind, unit_elems=1024, min_8bit_size=4096)
    assert h.state.fp32_state == [n < 4096 for n in sizes]
    assert all(h.state.m[i].dtype == torch.float32 for i in range(4))
    res = h.run(forced=True)
    check_bars(res, kind, "bf16", forced=True)
    assert res.forced["m_excess"] <= 1 and res.forced["v_excess"] <= 1


def test_dyn8_with_master_weights():
    wl = workloads.mixed(RAGGED, param_dtype="bf16", groups=2, steps=5)
    h = Harness(wl, "dyn8", unit_elems=1024, master=True)
    res = h.run(forced=True)
    check_bars(res, "dyn8", "bf16", forced=True)


@pytest.mark.parametrize("kind", VARIANTS)
def test_variant_few_large_full_size(kind):
    h = Harness(workloads.few_large(), kind, sample=4096, grad_device="cuda",
                param_device_init="cuda")
    res = h.run(steps=3, forced=True)
    check_bars(res, kind, "f32", forced=True)
    assert _exact_code_fraction(h) > 0.999


def test_dyn8_llama3_8b_full_size():
    free, _ = torch.cuda.mem_get_info()
    if free / 2 ** 30 < 70:
        pytest.skip("needs 70 GiB free")
    wl = workloads.llama3_8b()
    h = Harness(wl, "dyn8", sample=2048, grad_device="cuda", param_device_init="cuda")
    res = h.run(steps=2, forced=True)
    check_bars(res, "dyn8", "bf16", forced=True)
    del h
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
def test_codec_bit_exact_with_zero_betas(kind):
    """With beta1 = beta2 = 0 the new moments are exactly fp32(g) and fp32(g*g),
    the values the oracle encodes, so every code and scale must agree bit for
    bit: a direct check of the kernel's encoder, over blocks spanning many
    decades, exact codebook midpoints and a zero block."""
    from compact_state_gb300.torch_adapter import AdamWState
    from oracle.adamw import CODECS
    from oracle import dynamic8
    rng = np.random.default_rng(21)
    n = 256 * 64
    g = (10.0 ** rng.uniform(-9, 0, n)) * np.where(rng.random(n) < 0.5, -1, 1)
    g = g.reshape(-1, 256)
    g[:, 0] = np.where(rng.random(g.shape[0]) < 0.5, 1.0, -1.0)    # block max |g| = 1
    g[1] = 0.0                                                        # a zero block
    g[2, 1:128] = dynamic8.SIGNED_MID                                 # exact codebook
    g[3, 1:128] = -dynamic8.SIGNED_MID                                # midpoints (ties)
    # exact linear-codec ties: max 127 * 2^-10 gives scale 2^-10, so
    # x = (k + 1/2) * 2^-10 divides to a half-integer (ties to even)
    g[4, 0] = 127.0 * 2.0 ** -10
    g[4, 1:255] = np.arange(-126.5, 126.6, 1.0) * 2.0 ** -10
    g[4, 255] = 0.5 * 2.0 ** -10
    g = g.reshape(-1).astype(np.float32)
    p = torch.zeros(n, dtype=torch.float32, device="cuda")
    gt = torch.from_numpy(g).cuda()
    st = AdamWState([p], [gt], kind)
    st.run([dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0)])
    torch.cuda.synchronize()
    (enc_m, _, _), (enc_v, _, _) = CODECS[kind]
    g64 = g.astype(np.float64)
    qm, sm = enc_m(g64)
    qv, sv = enc_v((g64 * g64).astype(np.float32).astype(np.float64))
    assert np.array_equal(st.m[0].cpu().numpy().view(np.uint8), qm.view(np.uint8))
    assert np.array_equal(st.v[0].cpu().numpy().view(np.uint8), qv.view(np.uint8))
    assert np.array_equal(st.m_scale[0].cpu().numpy(), sm)
    assert np.array_equal(st.v_scale[0].cpu().numpy(), sv)


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
def test_mixed_param_dtypes_in_one_8bit_plan(kind):
    """An 8-bit plan whose params are all 16-bit runs the kernel variant
    whose stage holds 2-byte params; a plan that also holds an fp32 tensor
    runs the general one. Both must give the same bits for the same tensors:
    the 16-bit tensors stepped in a mixed plan equal the same tensors stepped
    in a plan of their own, over ragged sizes and several steps."""
    from compact_state_gb300 import adamw_plan_create, tensor_desc
    from compact_state_gb300.torch_adapter import AdamWState
    from tests.parity_harness import _bits_equal
    sizes = [70001, 8192 * 3, 257, 4099, 1]
    wl16 = workloads.mixed(sizes, param_dtype="bf16", groups=2, steps=4)
    wl32 = workloads.mixed([30000, 5], param_dtype="f32", groups=2, steps=4)
    p16a = [workloads.init_param(wl16, i).reshape(-1).cuda() for i in range(len(sizes))]
    p16b = [x.clone() for x in p16a]
    p32 = [workloads.init_param(wl32, i).reshape(-1).cuda() for i in range(2)]
    g16 = [torch.zeros_like(x) for x in p16a]
    g32 = [torch.zeros_like(x) for x in p32]
    alone = AdamWState(p16a, g16, kind, [t.group for t in wl16.tensors])
    mixed = AdamWState(p16b + p32, g16 + g32, kind,
                       [t.group for t in wl16.tensors] + [t.group for t in wl32.tensors])
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl16.groups]
    for s in range(1, 5):
        for i in range(len(sizes)):
            g16[i].copy_(workloads.grad(wl16, i, s).reshape(-1))
        for i in range(2):
            g32[i].copy_(workloads.grad(wl32, i, s).reshape(-1))
        alone.run(groups)
        mixed.run(groups)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        assert _bits_equal(p16a[i], p16b[i]), i
        assert _bits_equal(alone.m[i], mixed.m[i]) and _bits_equal(alone.v[i], mixed.v[i]), i
        assert _bits_equal(alone.m_scale[i], mixed.m_scale[i]), i
        assert _bits_equal(alone.v_scale[i], mixed.v_scale[i]), i
    assert torch.equal(alone.step[:len(sizes)], mixed.step[:len(sizes)])


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
def test_16bit_plan_with_small_units_matches_one_without(kind):
    """A 16-bit-param 8-bit plan whose work units are all large runs the
    16-bit kernel that never packs; adding small tensors switches the plan to
    the one that packs them several to a stage. The large tensors must get
    the same bits from both, over several steps."""
    from compact_state_gb300.torch_adapter import AdamWState
    from tests.parity_harness import _bits_equal
    big, small = [70001, 24576], [300, 7, 1500, 16]
    wl = workloads.mixed(big + small, param_dtype="bf16", groups=2, steps=3)
    pa = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(big))]
    pb = [x.clone() for x in pa]
    ps = [workloads.init_param(wl, len(big) + i).reshape(-1).cuda() for i in range(len(small))]
    ga = [torch.zeros_like(x) for x in pa]
    gs = [torch.zeros_like(x) for x in ps]
    grp = [t.group for t in wl.tensors]
    lean = AdamWState(pa, ga, kind, grp[:len(big)])
    packing = AdamWState(pb + ps, ga + gs, kind, grp)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    for s in range(1, 4):
        for i in range(len(big) + len(small)):
            (ga + gs)[i].copy_(workloads.grad(wl, i, s).reshape(-1))
        lean.run(groups)
        packing.run(groups)
    torch.cuda.synchronize()
    for i in range(len(big)):
        assert _bits_equal(pa[i], pb[i]), i
        assert _bits_equal(lean.m[i], packing.m[i]) and _bits_equal(lean.v[i], packing.v[i]), i
        assert _bits_equal(lean.m_scale[i], packing.m_scale[i]), i
        assert _bits_equal(lean.v_scale[i], packing.v_scale[i]), i
    assert torch.equal(lean.step[:len(big)], packing.step[:len(big)])


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
def test_codec_bit_exact_many_scales(kind):
    """As the test above, with block maxima spread over many decades (the
    codebook divides by them without an IEEE division per element), with
    quotients placed at and one ulp beside every codebook midpoint, and with
    scales that take the IEEE path (below 2^-64, and an all-ones
    significand): every code and scale equals the oracle's, bit for bit."""
    from compact_state_gb300.torch_adapter import AdamWState
    from oracle.adamw import CODECS
    from oracle import dynamic8
    rng = np.random.default_rng(99)
    nblk = 4096
    s = (rng.uniform(1.0, 2.0, nblk) * 2.0 ** rng.integers(-40, 10, nblk)).astype(np.float32)
    s[0] = np.float32(2.0 ** -70)                                 # IEEE path: tiny scale
    s[1] = np.uint32(0x3FFFFFFF).view(np.float32)                 # all-ones significand
    mids = np.concatenate([dynamic8.SIGNED_MID, dynamic8.UNSIGNED_MID]).astype(np.float32)
    mids = mids[np.isfinite(mids) & (mids > 0) & (mids < 1)]
    targets = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                              np.nextafter(mids, np.float32(2))])
    # quotients at and beside the midpoints, and 30% spread over eight decades
    t = rng.choice(targets, (nblk, 256)).astype(np.float32)
    spread = rng.random((nblk, 256)) < 0.3
    t[spread] = (10.0 ** rng.uniform(-8, 0, int(spread.sum()))).astype(np.float32)
    sign = np.where(rng.random((nblk, 256)) < 0.5, -1.0, 1.0).astype(np.float32)
    g = (t.astype(np.float64) * s[:, None].astype(np.float64)).astype(np.float32) * sign
    g[:, 0] = s * sign[:, 0]                                      # the block's max |g| is s
    g = np.clip(g, -s[:, None], s[:, None]).reshape(-1).astype(np.float32)
    n = g.size
    p = torch.zeros(n, dtype=torch.float32, device="cuda")
    gt = torch.from_numpy(g).cuda()
    st = AdamWState([p], [gt], kind)
    st.run([dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0)])
    torch.cuda.synchronize()
    (enc_m, _, _), (enc_v, _, _) = CODECS[kind]
    g64 = g.astype(np.float64)
    qm, sm = enc_m(g64)
    qv, sv = enc_v((g64 * g64).astype(np.float32).astype(np.float64))
    assert np.array_equal(st.m_scale[0].cpu().numpy(), sm)
    assert np.array_equal(st.v_scale[0].cpu().numpy(), sv)
    assert np.array_equal(st.m[0].cpu().numpy().view(np.uint8), qm.view(np.uint8))
    assert np.array_equal(st.v[0].cpu().numpy().view(np.uint8), qv.view(np.uint8))
