"""Pins for the oracle's expert FFN, FinalizeRouting and shared-expert add.

Sources: "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 一
(expert FFN intermediate 1536, 1 shared expert) and section 8.5 (routed path,
combine add, shared expert independent of gating); "HunyuanImage-3.0 MoE 多流
变体实战", 源码级实现拆解 §3 (output = hidden_states_mlp + combined_output).

The pins: a hand-worked example, the one-expert case against numpy's matmul
(a library routine), invariances (unselected experts, token order, duplicate
tokens), scaling=0 leaving only the shared expert, and linearity in the
routed weights.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def test_worked_example(golden_dir):
    rows = {}
    for line in open(f"{golden_dir}/swiglu_worked_example.txt"):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        rows[k] = [float(a) for a in v]
    x = _bf16([rows["x"]])
    wg = _bf16([rows["w_gate"]])
    wu = _bf16([rows["w_up"]])
    wd = _bf16(np.array(rows["w_down"])[:, None])
    y = oracle.swiglu_mlp(x, wg, wu, wd)
    np.testing.assert_allclose(y[0], rows["y"], rtol=1e-15)
    # Swapping gate and up changes the answer (silu is not symmetric): 2*silu(... )
    y_sw = oracle.swiglu_mlp(x, wu, wg, wd)
    assert not np.allclose(y_sw, y)


def _numpy_swiglu(x, wg, wu, wd):
    g = _f64(x) @ _f64(wg).T
    u = _f64(x) @ _f64(wu).T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ _f64(wd).T


def test_one_expert_layer_is_dense_swiglu_against_numpy_matmul():
    sh = synth.MoEShape("one", T=12, H=64, E=1, K=1, I=96, I_shared=0, scaling=1.0)
    x, logits = synth.make_activations(sh, seed=5)
    w = synth.make_weights(sh, seed=5, std=0.1)
    out, idx, tw = oracle.layer_forward(x, logits, w["w_gate"], w["w_up"], w["w_down"], K=1, scaling=1.0)
    assert np.all(idx == 0) and np.all(tw == 1.0)
    ref = _numpy_swiglu(x, w["w_gate"][0], w["w_up"][0], w["w_down"][0])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.swiglu_mlp(x, w["w_gate"][0], w["w_up"][0], w["w_down"][0]), ref,
                               rtol=1e-12, atol=1e-12)


def _tiny(seed=0, **kw):
    sh = synth.WORKLOADS["tiny"].with_(**kw)
    x, logits = synth.make_activations(sh, seed=seed)
    w = synth.make_weights(sh, seed=seed)
    return sh, x, logits, w


def _run(sh, x, logits, w, **kw):
    ws = (w.get("ws_gate"), w.get("ws_up"), w.get("ws_down"))
    return oracle.layer_forward(x, logits, w["w_gate"], w["w_up"], w["w_down"], *ws, K=sh.K,
                                scaling=kw.get("scaling", sh.scaling), route_norm=sh.route_norm,
                                tokens=kw.get("tokens"))


def test_layer_is_weighted_sum_of_expert_mlps_plus_shared_numpy():
    # Per token: sum_k w_k * MLP_{e_k}(x) + MLP_shared(x), each MLP by numpy matmul.
    sh, x, logits, w = _tiny(seed=1)
    out, idx, tw = _run(sh, x, logits, w)
    ref = _numpy_swiglu(x, w["ws_gate"], w["ws_up"], w["ws_down"])
    for t in range(sh.T):
        for k in range(sh.K):
            e = idx[t, k]
            ref[t] += tw[t, k] * _numpy_swiglu(x[t:t + 1], w["w_gate"][e], w["w_up"][e], w["w_down"][e])[0]
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_unselected_expert_weights_do_not_matter():
    sh, x, logits, w = _tiny(seed=2)
    logits[:, 3] = -50.0  # expert 3 never selected
    out, idx, _ = _run(sh, x, logits, w)
    assert not np.any(idx == 3)
    w2 = dict(w)
    for k in ("w_gate", "w_up", "w_down"):
        w2[k] = w[k].clone()
        w2[k][3] = 7.0
    out2, _, _ = _run(sh, x, logits, w2)
    assert np.array_equal(out, out2)
    # Changing a selected expert changes exactly the tokens routed to it.
    e = int(idx[0, 0])
    w3 = dict(w)
    w3["w_down"] = w["w_down"].clone()
    w3["w_down"][e] *= 2
    out3, _, _ = _run(sh, x, logits, w3)
    changed = np.any(out3 != out, axis=1)
    assert np.array_equal(changed, np.any(idx == e, axis=1))


def test_token_order_equivariance_and_duplicates():
    sh, x, logits, w = _tiny(seed=3)
    out, _, _ = _run(sh, x, logits, w)
    p = torch.randperm(sh.T, generator=torch.Generator().manual_seed(9))
    outp, _, _ = _run(sh, x[p], logits[p], w)
    np.testing.assert_allclose(outp, out[p.numpy()], rtol=1e-13, atol=1e-14)
    x2, l2 = x.clone(), logits.clone()
    x2[5], l2[5] = x2[2], l2[2]
    out2, _, _ = _run(sh, x2, l2, w)
    assert np.array_equal(out2[5], out2[2])
    # The subset API gives the same rows as the full call.
    sub, _, _ = _run(sh, x, logits, w, tokens=[7, 0, 7])
    np.testing.assert_allclose(sub, out[[7, 0, 7]], rtol=1e-13, atol=1e-14)


def test_scaling_zero_leaves_only_shared_expert():
    sh, x, logits, w = _tiny(seed=4)
    out0, _, _ = _run(sh, x, logits, w, scaling=0.0)
    shared = oracle.swiglu_mlp(x, w["ws_gate"], w["ws_up"], w["ws_down"])
    assert np.array_equal(out0, shared)


def test_linearity_in_routed_weights_and_no_shared():
    sh, x, logits, w = _tiny(seed=5)
    shared = oracle.swiglu_mlp(x, w["ws_gate"], w["ws_up"], w["ws_down"])
    o1, _, _ = _run(sh, x, logits, w, scaling=1.0)
    o3, _, _ = _run(sh, x, logits, w, scaling=3.0)
    np.testing.assert_allclose(o3 - shared, 3.0 * (o1 - shared), rtol=1e-12, atol=1e-12)
    w_ns = {k: v for k, v in w.items() if not k.startswith("ws_")}
    sh_ns = sh.with_(I_shared=0)
    o_ns, _, _ = oracle.layer_forward(x, logits, w["w_gate"], w["w_up"], w["w_down"], K=sh.K, scaling=1.0)
    np.testing.assert_allclose(o_ns, o1 - shared, rtol=1e-12, atol=1e-12)
    assert sh_ns.I_shared == 0 and set(w_ns) == {"w_gate", "w_up", "w_down"}


def test_bad_token_ids_rejected():
    sh, x, logits, w = _tiny()
    with pytest.raises(ValueError):
        _run(sh, x, logits, w, tokens=[sh.T])
