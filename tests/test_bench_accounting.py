"""Host-side accounting of bench.py (no GPU): the kernel-launch count a round
of the model workload reports must follow the decoder's sequencing.  The split
plans below are the ones the library reports on a 152-SM GB300 for the
8-layer model's products (vc_gemm_splits); with them the count equals the
1822 launches per timed round of the ncu launch list of the default model
bench (packed host cache)."""
import types

import bench

# (N, K, decode plan) -> K splits; > 1 means split (only whether a product is
# split, and whether its grid has more than 64 tiles, changes the count)
SPLITS = {
    (6144, 4096, True): 6, (4096, 4096, True): 8, (28672, 4096, True): 1, (4096, 14336, True): 9,
    (32000, 4096, True): 1,
    (6144, 4096, False): 2, (4096, 4096, False): 2, (28672, 4096, False): 1, (4096, 14336, False): 2,
    (32000, 4096, False): 1,
}


class FakeLib:
    @staticmethod
    def vc_gemm_splits(dt, N, K, decode):
        return SPLITS[(N, K, bool(decode))]


CFG = types.SimpleNamespace(n_layers=8, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, d_ff=14336,
                            vocab=32000)


def test_model_round_launch_count_matches_the_launch_list():
    assert bench.model_launches_per_round(CFG, FakeLib, packed=True) == 1822


def test_model_round_launch_count_parts():
    # a draft step: embedding, per layer q|k|v, RoPE (writing the ring), draft
    # attention, o, gate|up (SwiGLU epilogue), down; the LM head with its argmax
    # epilogue (normalising its rows), acceptance, the token scatter, the status fold
    draft = 1 + CFG.n_layers * 6 + 1 + 3
    # the verify forward: embedding, per layer RMSNorm, q|k|v (+ its reduction),
    # RoPE, verify attention and its combine, o (+ reduction), RMSNorm, gate|up,
    # down (+ reduction); the final RMSNorm, head, acceptance, status fold
    verify = 1 + CFG.n_layers * (2 + 4 + 1 + 2 + 3) + 1 + 1 + 2
    commit = CFG.n_layers + 1                      # ring appends with re-quantisation, host write-back
    expansion = 2 * CFG.n_layers                   # packed rows expanded, K and V per layer
    assert bench.model_launches_per_round(CFG, FakeLib, packed=True) == 32 * draft + verify + commit + expansion
    # keys rotated on the way into the cache: the ring append comes back in draft steps
    assert (bench.model_launches_per_round(CFG, FakeLib, packed=True, rotate=True) ==
            bench.model_launches_per_round(CFG, FakeLib, packed=True) + 32 * CFG.n_layers)
    assert (bench.model_launches_per_round(CFG, FakeLib, packed=False) ==
            bench.model_launches_per_round(CFG, FakeLib, packed=True) - expansion)
