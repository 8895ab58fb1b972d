"""GPU parity of the KIVI quantizer (vc_quantize_kv, vc_qcache_append): the
packed records, read back through the oracle's own record reader, must equal
the oracle's quantization bit for bit (codes, fp16 scales and zeros), and the
full-precision ring must hold the residual tokens."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import f32, lib

pytestmark = pytest.mark.gpu


def _check_cache(vc, cache, k, v, L, bits, R, bs=None, hs=None, rotate=False):
    B, H, _, d = k.shape
    G = 32
    nq = ((L - R) // G) * G if L - R > 0 else 0
    bs = list(range(B)) if bs is None else list(bs)
    hs = list(range(H)) if hs is None else list(hs)
    kq = f32(k[bs][:, hs, :L])
    vq = f32(v[bs][:, hs, :L])
    ref = oracle.kivi_quantize(kq, vq, bits, G, R, rotate=rotate, rotate_bf16=k.dtype == torch.bfloat16)
    recs = cache.record_view().cpu().numpy()
    for i, b in enumerate(bs):
        for j, h in enumerate(hs):
            if nq:
                got = oracle.unpack_records(recs[b, h, :nq // G], bits, d)
                assert np.array_equal(got["kcode"], ref["kcode"][i, j]), (b, h)
                assert np.array_equal(got["vcode"], ref["vcode"][i, j]), (b, h)
                assert np.array_equal(got["kscale"], ref["kscale"][i, j]), (b, h)
                assert np.array_equal(got["kzero"], ref["kzero"][i, j]), (b, h)
                assert np.array_equal(got["vscale"], ref["vscale"][i, j]), (b, h)
                assert np.array_equal(got["vzero"], ref["vzero"][i, j]), (b, h)
    # residual ring
    kr = f32(cache.k_res)
    for i, b in enumerate(bs):
        for j, h in enumerate(hs):
            for p in range(nq, L):
                assert np.array_equal(kr[b, h, p % cache.res_cap], ref["kres"][i, j, p - nq])
    assert cache.n_groups.cpu().tolist() == [nq // G] * B
    assert cache.seq_len.cpu().tolist() == [L] * B


@pytest.mark.parametrize("bits,d,R,L,dtype,rotate", [
    (2, 128, 128, 300, torch.bfloat16, False),     # several groups + ragged residual
    (4, 128, 0, 256, torch.bfloat16, False),
    (4, 64, 0, 517, torch.float32, False),         # tiny-decoder shape, fp32
    (2, 64, 16, 40, torch.float32, False),         # one group
    (2, 128, 128, 100, torch.bfloat16, False),     # shorter than the window: no group
    (2, 128, 128, 300, torch.bfloat16, True),      # rotated keys
    (4, 64, 16, 517, torch.float32, True),
    (2, 128, 64, 100, torch.bfloat16, True),
])
def test_quantize_matches_oracle(bits, d, R, L, dtype, rotate):
    vc = lib()
    B, H = 3, 2
    k, v = inputs.kv_with_outliers(B, H, L + 5, d, seed=11 + bits + d, device="cuda", dtype=dtype)
    G = 32
    maxg = max(1, (L - R) // G + 1)
    cache = vc.QCache(B, H, d, bits, maxg, R + G + 8, R, res_dtype=dtype, rotate=rotate)
    vc.vc_quantize_kv(k.contiguous(), v.contiguous(), cache, L=L)
    torch.cuda.synchronize()
    _check_cache(vc, cache, k, v, L, bits, R, rotate=rotate)


@pytest.mark.parametrize("bits,d", [(2, 128), (4, 128), (2, 64)])
def test_quantize_codes_at_half_integers(bits, d):
    """Every group spans [0, qmax * 2^j] (K: tokens 0 and 1 of each channel;
    V: channels 0 and 1 of each 32-channel group), so its scale is exactly 2^j
    and the other values, drawn from the multiples of 2^(j-1), put x / s on
    integers and on ties (rint: ties to even).  Every word holding a tie takes
    the quantizer's exact-quotient path; the records must still equal the
    oracle's bit for bit."""
    vc = lib()
    B, H, L, G = 2, 2, 96, 32
    qmax = (1 << bits) - 1
    rng = np.random.default_rng(7 + bits + d)
    halves = rng.integers(0, 2 * qmax + 1, size=(2, B, H, L, d)).astype(np.float32) * 0.5
    halves[0, :, :, 0::G, :] = 0.0
    halves[0, :, :, 1::G, :] = qmax
    halves[1, :, :, :, 0::G] = 0.0
    halves[1, :, :, :, 1::G] = qmax
    scale = np.array([0.125, 1.0, 4.0, 0.5], dtype=np.float32).reshape(B, H, 1, 1)
    k = torch.from_numpy(halves[0] * scale).to(torch.bfloat16).cuda()
    v = torch.from_numpy(halves[1] * scale).to(torch.bfloat16).cuda()
    assert torch.equal(k.float().cpu(), torch.from_numpy(halves[0] * scale))   # exact in bf16
    cache = vc.QCache(B, H, d, bits, L // G, G + 8, 0)
    vc.vc_quantize_kv(k, v, cache, L=L)
    torch.cuda.synchronize()
    _check_cache(vc, cache, k, v, L, bits, 0)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("bits,R,rotate", [(2, 128, False), (4, 0, False), (2, 64, True)])
def test_append_equals_one_shot(bits, R, rotate):
    """Appending tokens (ragged per sequence) and re-quantizing leaving groups
    gives the same records (and ring) as quantizing the whole sequence at once."""
    vc = lib()
    B, H, d, G = 3, 2, 128, 32
    L0, adds = 200, [[17, 0, 40], [33, 50, 1], [0, 12, 30]]
    total = L0 + max(sum(a[b] for a in adds) for b in range(B))
    k, v = inputs.kv_with_outliers(B, H, total + 1, d, seed=21, device="cuda")
    maxg = total // G + 1
    cache = vc.QCache(B, H, d, bits, maxg, R + G + 64, R, rotate=rotate)
    vc.vc_quantize_kv(k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), cache)
    lens = [L0] * B
    for a in adds:
        m = max(a)
        kn = torch.zeros(B, H, max(m, 1), d, dtype=k.dtype, device="cuda")
        vn = torch.zeros_like(kn)
        for b in range(B):
            kn[b, :, :a[b]] = k[b, :, lens[b]:lens[b] + a[b]]
            vn[b, :, :a[b]] = v[b, :, lens[b]:lens[b] + a[b]]
            lens[b] += a[b]
        vc.vc_qcache_append(cache, kn, vn, torch.tensor(a, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.seq_len.cpu().tolist() == lens
    assert int(cache.status.item()) == 0
    for b in range(B):
        L = lens[b]
        nq = ((L - R) // G) * G if L > R else 0
        assert int(cache.n_groups[b]) == nq // G
        ref = oracle.kivi_quantize(f32(k[b:b + 1, :, :L]), f32(v[b:b + 1, :, :L]), bits, G, R, rotate=rotate)
        recs = cache.record_view().cpu().numpy()
        ring = f32(cache.k_res)
        for h in range(H):
            got = oracle.unpack_records(recs[b, h, :nq // G], bits, d)
            assert np.array_equal(got["kcode"], ref["kcode"][0, h])
            assert np.array_equal(got["kscale"], ref["kscale"][0, h])
            assert np.array_equal(got["vscale"], ref["vscale"][0, h])
            assert np.array_equal(got["kzero"], ref["kzero"][0, h])
            for p in range(nq, L):
                assert np.array_equal(ring[b, h, p % cache.res_cap], ref["kres"][0, h, p - nq])


def test_append_without_requantize_then_rollback():
    vc = lib()
    B, H, d, G, R = 2, 1, 64, 32, 0
    k, v = inputs.kv_with_outliers(B, H, 128, d, seed=5, device="cuda", dtype=torch.float32)
    cache = vc.QCache(B, H, d, 4, 4, 64, R, res_dtype=torch.float32)
    vc.vc_quantize_kv(k[:, :, :64].contiguous(), v[:, :, :64].contiguous(), cache)
    kn = k[:, :, 64:80].contiguous()
    vn = v[:, :, 64:80].contiguous()
    vc.vc_qcache_append(cache, kn, vn, torch.tensor([16, 5], dtype=torch.int32, device="cuda"),
                        requantize=False)
    torch.cuda.synchronize()
    assert cache.seq_len.cpu().tolist() == [80, 69] and cache.n_groups.cpu().tolist() == [2, 2]
    ring = f32(cache.k_res)
    assert np.array_equal(ring[0, 0, 0:16], f32(k[0, 0, 64:80]))      # positions 64.. at slot p % 64
    assert np.array_equal(ring[1, 0, 0:5], f32(k[1, 0, 64:69]))
    # overflowing the ring is reported and clamped, not written out of bounds
    big = torch.zeros(B, H, 80, d, dtype=torch.float32, device="cuda")
    vc.vc_qcache_append(cache, big, big, torch.tensor([80, 0], dtype=torch.int32, device="cuda"),
                        requantize=False)
    torch.cuda.synchronize()
    assert int(cache.status.item()) != 0
    assert int(cache.seq_len[0]) - int(cache.n_groups[0]) * G <= cache.res_cap


def test_full_size_draft_workload_sampled():
    """The 16 x 8 x 32768 x 128 2-bit cache (R = 128): records of sampled
    (sequence, head) pairs against the oracle."""
    vc = lib()
    B, H, L, d, R = 16, 8, 32768, 128, 128
    k, v = inputs.kv_with_outliers(B, H, L, d, seed=2, device="cuda")
    cache = vc.QCache(B, H, d, 2, (L - R) // 32, R + 64, R)
    vc.vc_quantize_kv(k, v, cache)
    torch.cuda.synchronize()
    _check_cache(vc, cache, k, v, L, 2, R, bs=[0, 9, 15], hs=[0, 5])
