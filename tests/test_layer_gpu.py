"""One MoE layer forward through the whole library, against the oracle.

plan -> dispatch -> prefetch of both projections' weights -> grouped GEMM
(H -> H') -> grouped GEMM (H' -> H) -> combine: the static buffer flows
through the two expert projections and back ("月之暗面开源MoonEP：面向MoE训练的
专家并行通信库", sections 核心技术 and 内存契约与权重布局). The oracle composes
the same steps (each product exact in double, rounded to bf16 like the
kernel). Hidden states and weights are small integers, so every product sum
is an integer below 2^24, exact in fp32 in any order: the layer output must
match bit for bit, for the training plan and for the inference fallback.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


def _int_bf16(shape, seed, tag, lo=-2, hi=2):
    return oracle.f32_to_bf16(synth.integer_valued(shape, seed, lo, hi, tag=tag))


def _round_bf16(y64):
    return oracle.f32_to_bf16(y64.astype(np.float32))


@pytest.mark.parametrize("fallback", [False, True], ids=["train", "inference_fallback"])
def test_layer_forward_matches_oracle(fallback):
    s = synth.Shape(R=4, E=16, K=4, S=256, H=256, B=4 if not fallback else 1)
    Hp = 128
    idx, w = synth.routing(s, seed=7, alpha=1.5)
    ref = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B, fallback=fallback)
    assert ref["status"] == "ok"
    hidden = _int_bf16((s.N, s.H), 7, 80)
    w1 = _int_bf16((s.E, s.H, Hp), 7, 81)
    w2 = _int_bf16((s.E, Hp, s.H), 7, 82, lo=-1, hi=1)

    # GPU: the library end to end
    plan_fn = mep.mep_plan_remote_fallback if fallback else mep.mep_plan
    p = plan_fn(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    buf = mep.mep_dispatch(to_dev(hidden), p.dst_pos, p.status, s.R, s.S, s.K)
    w1_d, w2_d = to_dev(w1), to_dev(w2)
    s1 = torch.zeros((s.R, s.B, s.H, Hp), dtype=torch.bfloat16, device=DEV)
    s2 = torch.zeros((s.R, s.B, Hp, s.H), dtype=torch.bfloat16, device=DEV)
    mep.mep_prefetch(p.slot_expert, w1_d, s1, p.status, s.E)
    mep.mep_prefetch(p.slot_expert, w2_d, s2, p.status, s.E)
    h1 = mep.mep_grouped_gemm(buf, p.cu_seqlens, w1_d, s1, p.status, s.R, s.S, s.K)
    y = mep.mep_grouped_gemm(h1, p.cu_seqlens, w2_d, s2, p.status, s.R, s.S, s.K)
    out = mep.mep_combine(y, to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0

    # oracle: the same composition
    buf_r = oracle.dispatch(hidden, ref["dst_pos"], s.A)
    used = ref["slot_expert"] >= 0
    s1_r = np.zeros((s.R, s.B, s.H, Hp), np.uint16)
    s2_r = np.zeros((s.R, s.B, Hp, s.H), np.uint16)
    s1_r[used] = w1[ref["slot_expert"][used]]
    s2_r[used] = w2[ref["slot_expert"][used]]
    h1_r = _round_bf16(oracle.grouped_gemm(buf_r, ref["cu_seqlens"], w1, s1_r))
    y_r = _round_bf16(oracle.grouped_gemm(h1_r, ref["cu_seqlens"], w2, s2_r))
    out_r = oracle.combine(y_r, w, ref["dst_pos"])

    np.testing.assert_array_equal(to_np(p.cu_seqlens), ref["cu_seqlens"])
    np.testing.assert_array_equal(to_np(h1), h1_r)
    np.testing.assert_array_equal(to_np(y), y_r)
    np.testing.assert_array_equal(to_np(out), out_r)
