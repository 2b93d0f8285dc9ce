"""GPU parity of gdn_prefill_backward against the oracle's backward pass
(itself pinned to finite differences of the forward oracle): every gradient
at the fp32 tolerance (the backward kernels compute in fp32 whatever the stream
dtype; bf16 streams are read exactly), element by element for the per-token
gradients and the initial state's, normwise for the parameter gradients that
sum over every token and head (tests.helpers.parity_sum)."""
import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import parity, parity_sum, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# gradients that are sums over every token and head: checked normwise (tests.helpers.parity_sum)
SUMMED = ("conv_w", "A_log", "dt_bias", "norm_w")
KEYS = {"q": "x_q", "k": "x_k", "v": "x_v", "a": "a", "b": "b", "z": "z", "conv_w": "conv_w", "A_log": "A_log",
        "dt_bias": "dt_bias", "norm_w": "norm_w", "init_state": "init_state"}


def _check_backward(cfg, with_dfinal=True, slow_decay=False):
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    bf16 = cfg.dtype == "bf16"
    inp = synth.make_prefill(cfg)
    if slow_decay:                     # gradients flow back through many steps of the state
        inp["dt_bias"][:] = -3.0
    rng = np.random.default_rng(cfg.seed + 7)
    dy = rng.standard_normal((cfg.T, cfg.h_v, cfg.d_v)).astype(np.float32)
    if bf16:
        dy = synth.round_bf16(dy)
    dfinal = rng.standard_normal((cfg.N, cfg.h_v, cfg.d_k, cfg.d_v)).astype(np.float32) if with_dfinal else None
    t = to_torch(inp, bf16)
    dy_t = torch.from_numpy(dy).to("cuda", torch.bfloat16 if bf16 else torch.float32)
    df_t = None if dfinal is None else torch.from_numpy(dfinal).cuda()
    g = gdn.prefill_backward(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                             t["dt_bias"], t["norm_w"], t["cu_seqlens"], dy_t, t.get("init_state"), df_t)
    torch.cuda.synchronize()
    r = ref.prefill_backward(inp, inp["cu_seqlens"], dy, inp["init_state"], dfinal)
    for name, key in KEYS.items():
        check = parity_sum if name in SUMMED else parity
        check(g[name].cpu().numpy(), r[key], "fp32", f"d{name}")


@pytest.mark.parametrize("case", ["tiny_fp32", "bf16_d128_varlen", "fp32_d32_gqa4", "bf16_slow_decay",
                                  "bf16_dk128_dv64", "fp32_dk64_dv128"])
def test_backward_matches_oracle(case):
    if case == "tiny_fp32":
        cfg = synth.scaled(synth.TINY, init_std=0.05)
        _check_backward(cfg)
    elif case == "bf16_d128_varlen":          # several 32-token blocks, ragged ends, an empty sequence
        cfg = synth.scaled(synth.VARLEN_32K, lengths=(100, 0, 33, 64), h_qk=2, h_v=4, init_std=0.02, seed=61)
        _check_backward(cfg)
    elif case == "fp32_d32_gqa4":
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(70, 5), h_qk=1, h_v=4, d_k=32, d_v=32, dtype="fp32",
                           init_std=0.02, seed=62)
        _check_backward(cfg, with_dfinal=False)
    elif case == "bf16_slow_decay":
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(160,), h_qk=1, h_v=2, init_std=0.02, seed=63)
        _check_backward(cfg, slow_decay=True)
    elif case == "bf16_dk128_dv64":          # the d_k = 128 forms of the forward and reverse kernels, 2 slices
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(100, 37), h_qk=1, h_v=2, d_k=128, d_v=64, init_std=0.02,
                           seed=64)
        _check_backward(cfg)
    else:                                    # their general forms with d_v = 128 (4 slices)
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(70,), h_qk=1, h_v=2, d_k=64, d_v=128, dtype="fp32",
                           init_std=0.02, seed=65)
        _check_backward(cfg)


@pytest.mark.slow
def test_backward_full_heads_1024_tokens():
    """16 q/k heads, 32 value heads, d = 128, bf16, two sequences (1024 tokens in all)."""
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(700, 324), init_std=0.02, seed=64)
    _check_backward(cfg)
