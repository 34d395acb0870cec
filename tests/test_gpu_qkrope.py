"""GPU parity of the fused Q/K RMSNorm + rotary embedding producer
(``sab_qk_norm_rope``) against the fp64 oracle (``oracle/qkrope.py``), and of
its fused ring append (BF16 ring: the slot holds exactly k' and v; FP8 ring:
the codes and scales equal the oracle quantiser applied to k' and v).

Tolerance: the kernel computes in fp32 and rounds to bf16 once, so each
output lies within one bf16 unit in the last place (2^-8 relative) of the
exact value, plus fp32 trigonometry and angle rounding (< 1e-5 absolute at
these positions)."""

import numpy as np
import pytest
import torch

from oracle import fp8 as OF
from oracle import qkrope as OQ
from streaming_attention_block_gb300 import KVRing, RopeDesc, synth
import streaming_attention_block_gb300 as sab

from tests._common import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sab.library()


def _within_one_ulp(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{what}: {len(bad)} outside one bf16 ulp, max err {err.max():.3e}, first {bad[:3]}"


CASES = [
    # (B, H, D, grid (F, Hp, Wp), bands (t, h, w), chunk, gammas)
    ("wan_bands", 1, 3, 128, (2, 4, 6), (44, 42, 42), 5, True),
    ("one_dim", 2, 2, 64, (40, 1, 1), (64, 0, 0), 3, False),
    ("frames_only", 1, 4, 128, (3, 2, 2), (128, 0, 0), 0, True),
]


@pytest.mark.parametrize("name,B,H,D,grid,bands,chunk,gam", CASES, ids=[c[0] for c in CASES])
def test_qk_norm_rope_matches_oracle(name, B, H, D, grid, bands, chunk, gam):
    Lc = grid[0] * grid[1] * grid[2]
    w = synth.Workload("r", B=B, H=H, D=D, Lc=Lc, R=2, W=1, seed=91)
    gen = synth.generator(91)
    q, k, v = synth.chunk_qkv(w, gen)
    gq = gk = None
    if gam:
        gq = (0.5 + torch.rand(H * D, generator=gen)).float()
        gk = (0.5 + torch.rand(H * D, generator=gen)).float()
    ring = KVRing(1, B, H, D, Lc, 2)
    rope = RopeDesc(*grid, *bands, 10000.0, 1e-6)
    Qo, Ko, Vo = (torch.empty_like(x, device="cuda") for x in (q, k, v))
    sab.qk_norm_rope(ring.handle, 0, chunk, q.cuda(), k.cuda(), v.cuda(), rope, Qo, Ko, Vo,
                     gamma_q=None if gq is None else gq.cuda(), gamma_k=None if gk is None else gk.cuda())
    torch.cuda.synchronize()
    rq, rk = OQ.qk_norm_rope(f32(q), f32(k), chunk, grid, bands, None if gq is None else gq.numpy(),
                             None if gk is None else gk.numpy())
    _within_one_ulp(Qo, rq, f"{name} q'")
    _within_one_ulp(Ko, rk, f"{name} k'")
    assert torch.equal(Vo.cpu(), v), f"{name}: v must pass through bit-exact"


@pytest.mark.parametrize("kv_dtype", [sab.KV_BF16, sab.KV_FP8_E4M3], ids=["bf16_ring", "fp8_ring"])
def test_fused_append_writes_k_prime_and_v(kv_dtype):
    B, H, D, grid, bands = 1, 2, 128, (2, 8, 8), (44, 42, 42)
    Lc, R = 128, 3
    w = synth.Workload("r", B=B, H=H, D=D, Lc=Lc, R=R, W=1, seed=92)
    gen = synth.generator(92)
    ring = KVRing(1, B, H, D, Lc, R, kv_dtype=kv_dtype)
    rope = RopeDesc(*grid, *bands, 10000.0, 1e-6)
    for c in range(R + 2):
        q, k, v = (x.cuda() for x in synth.chunk_qkv(w, gen))
        Qo, Ko, Vo = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        sab.qk_norm_rope(ring.handle, 0, c, q, k, v, rope, Qo, Ko, Vo, append=True)
        torch.cuda.synchronize()
        assert ring.slot_of(0, c) == c % R
        K, V, KS, VS = ring.layer_views(0)
        rows = slice((c % R) * Lc, (c % R + 1) * Lc)
        if kv_dtype == sab.KV_BF16:
            assert torch.equal(K[:, :, rows].cpu(), Ko.permute(0, 2, 1, 3).cpu()), f"chunk {c}: ring K != k'"
            assert torch.equal(V[:, :, rows].cpu(), v.permute(0, 2, 1, 3).cpu()), f"chunk {c}: ring V != v"
        else:
            kc, ks = OF.quantize_chunk_bhld(f32(Ko.cpu()))
            vc, vs = OF.quantize_chunk_bhld(f32(v.cpu()))
            assert np.array_equal(K[:, :, rows].cpu().numpy(), kc) and np.array_equal(KS[:, :, c % R].cpu().numpy(), ks)
            assert np.array_equal(V[:, :, rows].cpu().numpy(), vc) and np.array_equal(VS[:, :, c % R].cpu().numpy(), vs)
    with pytest.raises(sab.SabError) as e:  # chunk order is enforced when appending
        sab.qk_norm_rope(ring.handle, 0, R + 5, q, k, v, rope, Qo, Ko, Vo, append=True)
    assert e.value.status == 3


def test_invalid_rope_descriptions():
    ring = KVRing(1, 1, 2, 128, 48, 2)
    q = torch.zeros((1, 48, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    for bad in (RopeDesc(2, 4, 5, 44, 42, 42, 10000.0, 1e-6),   # grid != chunk_tokens
                RopeDesc(2, 4, 6, 43, 43, 42, 10000.0, 1e-6),   # odd bands
                RopeDesc(2, 4, 6, 44, 42, 40, 10000.0, 1e-6),   # bands do not sum to D
                RopeDesc(2, 4, 6, 44, 42, 42, 1.0, 1e-6),       # base <= 1
                RopeDesc(2, 4, 6, 44, 42, 42, 10000.0, 0.0)):   # eps <= 0
        with pytest.raises(sab.SabError) as e:
            sab.qk_norm_rope(ring.handle, 0, 0, q, q, q, bad, out)
        assert e.value.status == 1
    fp8 = KVRing(1, 1, 2, 128, 48, 2, kv_dtype=sab.KV_FP8_E4M3)
    with pytest.raises(sab.SabError) as e:  # an 8-bit ring needs K_out and V_out to append
        sab.qk_norm_rope(fp8.handle, 0, 0, q, q, q, RopeDesc(2, 4, 6, 44, 42, 42, 10000.0, 1e-6), out, append=True)
    assert e.value.status == 1
