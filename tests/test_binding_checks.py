"""The Python binding refuses tensors the C ABI would misread (it sees only
pointers): wrong dtype, wrong shape or layout, non-contiguous, or host
memory.  Every check runs before the library is called, so these tests need
no GPU."""
import dataclasses

import pytest
import torch

from block_diffusion_lm_gb300 import csbp
from block_diffusion_lm_gb300.inputs import WORKLOADS, make_inputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_diffusion_lm_gb300 import build
    build.build()


def attn_case(has_clean=True):
    w = WORKLOADS["tiny"]
    attn = csbp.BlockDiffusionAttention(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d,
                                        has_clean_queries=has_clean, device="cpu")
    t = make_inputs(w, "cpu")
    if not has_clean:
        t["q_clean"] = t["do_clean"] = None
    return attn, t


def test_host_tensors_are_refused():
    attn, t = attn_case()
    with pytest.raises(ValueError, match="q_clean must be a CUDA tensor"):
        attn.forward(t)


@pytest.mark.parametrize("name,bad,msg", [
    ("q_corr", lambda x: x.float(), "q_corr must be torch.bfloat16"),
    ("k_clean", lambda x: x.transpose(1, 2).contiguous(), "k_clean must have shape"),
    ("v_corr", lambda x: x.transpose(1, 2).contiguous().transpose(1, 2),
     "v_corr must have contiguous heads and features"),
    ("k_corr", lambda x: x.transpose(2, 3).contiguous().transpose(2, 3),
     "k_corr must have contiguous heads"),
    ("q_clean", lambda x: None, "q_clean is required"),
])
def test_forward_inputs_are_checked(name, bad, msg):
    attn, t = attn_case()
    t[name] = bad(t[name])
    with pytest.raises(ValueError, match=msg):
        attn.forward(t)


def test_packed_qkv_views_pass_the_layout_checks():
    """q, k and v as views into one packed [batch][L][Hq + 2 Hkv][d] tensor
    per copy (token stride (Hq + 2 Hkv) d) get as far as the device check;
    outputs and dO must still be contiguous."""
    attn, t = attn_case()
    w = WORKLOADS["tiny"]
    for copy in ("clean", "corr"):
        packed = torch.cat([t[f"q_{copy}"], t[f"k_{copy}"], t[f"v_{copy}"]], dim=2)
        t[f"q_{copy}"] = packed[:, :, :w.Hq]
        t[f"k_{copy}"] = packed[:, :, w.Hq:w.Hq + w.Hkv]
        t[f"v_{copy}"] = packed[:, :, w.Hq + w.Hkv:]
        assert not t[f"k_{copy}"].is_contiguous()
    with pytest.raises(ValueError, match="q_clean must be a CUDA tensor"):
        attn.forward(t)
    inp = csbp._inputs(t)
    assert list(inp.stride_tok) == [(w.Hq + 2 * w.Hkv) * w.d] * 6
    oc, ox, lse = attn.alloc_outputs()
    with pytest.raises(ValueError, match="o_corr must be contiguous"):
        attn.forward(t, out=(oc, ox.transpose(1, 2).contiguous().transpose(1, 2), lse))


def test_broadcast_views_are_refused():
    """A zero stride means "contiguous" to the library, so an expanded
    (stride-0) batch or token dimension must not reach it."""
    w = WORKLOADS["tiny"]
    attn = csbp.BlockDiffusionAttention(2, w.L, w.M, w.Hq, w.Hkv, w.d, device="cpu")
    t = make_inputs(dataclasses.replace(w, batch=2), "cpu")
    t["k_clean"] = t["k_clean"][:1].expand(2, -1, -1, -1)
    with pytest.raises(ValueError, match="k_clean has a broadcast"):
        attn.forward(t)
    t = make_inputs(dataclasses.replace(w, batch=2), "cpu")
    t["v_corr"] = t["v_corr"][:, :1].expand(-1, w.L, -1, -1)
    with pytest.raises(ValueError, match="v_corr has a broadcast"):
        attn.forward(t)


def test_sequence_first_layouts_are_refused_with_a_clear_message():
    """A [L][batch][H][d] tensor viewed as [batch][L][H][d] interleaves the
    batch entries; the library takes batch-first strides only."""
    w = WORKLOADS["tiny"]
    attn = csbp.BlockDiffusionAttention(2, w.L, w.M, w.Hq, w.Hkv, w.d, device="cpu")
    t = make_inputs(dataclasses.replace(w, batch=2), "cpu")
    t["q_corr"] = t["q_corr"].transpose(0, 1).contiguous().transpose(0, 1)
    with pytest.raises(ValueError, match="q_corr batch entries must not interleave"):
        attn.forward(t)


def test_forward_outputs_are_checked():
    attn, t = attn_case()
    oc, ox, lse = attn.alloc_outputs()
    with pytest.raises(ValueError, match="lse must have shape"):
        attn.forward(t, out=(oc, ox, lse[:, :1].contiguous()))
    with pytest.raises(ValueError, match="o_corr must be torch.bfloat16"):
        attn.forward(t, out=(oc, ox.float(), lse))


def test_backward_gradients_are_checked():
    attn, t = attn_case()
    out = attn.alloc_outputs()
    g = attn.alloc_grads()
    g["dk_corr"] = g["dk_corr"][:, :-1].contiguous()
    with pytest.raises(ValueError, match="dk_corr must have shape"):
        attn.backward(t, out, grads=g)
    g = attn.alloc_grads()
    t["do_corr"] = None
    with pytest.raises(ValueError, match="do_corr is required"):
        attn.backward(t, out, grads=g)


def test_clean_query_tensors_are_optional_without_clean_queries():
    """Without clean queries the clean-query tensors may be None; the clean
    K/V (read by the corrupted queries) are still required.  Validation then
    gets as far as the device check of the first tensor it meets."""
    attn, t = attn_case(has_clean=False)
    with pytest.raises(ValueError, match="k_clean must be a CUDA tensor"):
        attn.forward(t)
    t["k_clean"] = None
    with pytest.raises(ValueError, match="k_clean is required"):
        attn.forward(t)


def test_lse_merge_arguments_are_checked():
    o = [torch.zeros(10, 2, 64), torch.zeros(10, 2, 64)]
    z = [torch.zeros(2, 10), torch.zeros(2, 10)]
    o_out = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    z_out = torch.zeros(2, 10)
    with pytest.raises(ValueError, match="one LSE part per output part"):
        csbp.lse_merge(o, z[:1], o_out, z_out)
    with pytest.raises(ValueError, match=r"lse_parts\[1\] must have shape"):
        csbp.lse_merge(o, [z[0], z[1].T.contiguous()], o_out, z_out)
    with pytest.raises(ValueError, match="o_out must be torch.bfloat16"):
        csbp.lse_merge(o, z, o_out.float(), z_out)
    with pytest.raises(ValueError, match=r"o_parts\[0\] must be a CUDA tensor"):
        csbp.lse_merge(o, z, o_out, z_out)


def test_vocab_ce_arguments_are_checked():
    N, Dm, V = 130, 64, 256
    ce = csbp.VocabCrossEntropy(N, Dm, V, device="cpu")
    h = torch.zeros(N, Dm, dtype=torch.bfloat16)
    w = torch.zeros(V, Dm, dtype=torch.bfloat16)
    tgt = torch.zeros(N, dtype=torch.int32)
    with pytest.raises(ValueError, match="target must be torch.int32"):
        ce(h, w, tgt.long())
    with pytest.raises(ValueError, match="w must have shape"):
        ce(h, w.T.contiguous(), tgt)
    with pytest.raises(ValueError, match="h must be a CUDA tensor"):
        ce(h, w, tgt)
    frozen = csbp.VocabCrossEntropy(N, Dm, V, head_grad=False, device="cpu")
    loss, lse, dh, _ = frozen.alloc_outputs()
    with pytest.raises(ValueError, match="dw must be None for a frozen head"):
        frozen(h, w, tgt, out=(loss, lse, dh, torch.zeros(V, Dm)))
