"""The MoE FFN layer step captured once as a CUDA graph: replays give the eager step's bytes,
also after the inputs change in place between replays."""
import pytest
import torch

from mxfp8_block_scaled_rowwise_gb300 import synth
from mxfp8_block_scaled_rowwise_gb300.layer import MoEFFNStep
from gpu_util import check_dev_err, dev  # noqa: F401

pytestmark = pytest.mark.gpu

OUTS = ("out", "dx", "dgate", "dw1", "dw2", "out1", "h_q", "dh_q")


def _fill(st, seed):
    g = synth.generator(seed)
    st.x.copy_(synth.randn_bf16(st.x.shape, g))
    logits = torch.randn(st.T, st.E, generator=g)
    ids = synth.topk_ids(logits, st.k)
    st.ids.copy_(ids)
    st.gate.copy_(torch.softmax(logits.gather(1, ids.long()), dim=1))
    st.w1.copy_(synth.randn_bf16(st.w1.shape, g, std=st.H ** -0.5))
    st.w2.copy_(synth.randn_bf16(st.w2.shape, g, std=st.I ** -0.5))
    st.dout.copy_(synth.randn_bf16(st.dout.shape, g, std=1e-2))


def _snapshot(st):
    return {n: getattr(st, n).clone() for n in OUTS}


def test_graph_replay_matches_eager_step(dev):
    st = MoEFFNStep(384, 8, 3, 256, 128, device=dev)
    _fill(st, 71)
    st.step()                      # eager, also the warm-up the capture needs
    check_dev_err(st.dev_err)
    eager1 = _snapshot(st)
    graph = st.capture()
    for n in OUTS:
        getattr(st, n).zero_()
    graph.replay()
    check_dev_err(st.dev_err)
    for n in OUTS:
        assert torch.equal(getattr(st, n), eager1[n]), n
    # new inputs in place: the replay follows them, and equals a fresh eager step
    _fill(st, 72)
    graph.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(st)
    st.step()
    check_dev_err(st.dev_err)
    for n in OUTS:
        assert torch.equal(replayed[n], getattr(st, n)), n
        assert not torch.equal(replayed[n], eager1[n]), n
