"""GPU parity of pkv_philox_uniforms against the oracle's Philox-4x64-10
uniforms (bit-exact), and the sampler drawing from device-generated
uniforms: the same tokens as the oracle fed the oracle's uniforms."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import pkv, workloads

from parity import check_sampler

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("seed,offset,B", [(42, 0, 1), (42, 1, 256), (0, 0, 65535),
                                           (2**64 - 1, 2**64 - 1, 1000), (7, 123456789, 4097)])
def test_uniforms_match_oracle(seed, offset, B):
    got = pkv.philox_uniforms(seed, offset, B, device=DEV).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.uniforms(seed, offset, B))


def test_uniforms_in_a_graph_and_on_a_stream():
    out = torch.empty(512, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.philox_uniforms(42, 5, 512, out=out)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.philox_uniforms(42, 6, 512, out=out)
        g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.uniforms(42, 6, 512))


@pytest.mark.parametrize("name", ["pr1", "mixed"])
def test_sampler_with_device_uniforms(name):
    w = workloads.make(name) if name == "pr1" else workloads.mixed(B=64, V=32768)
    B = w.B
    u_dev = pkv.philox_uniforms(42, 3, B, device=DEV)
    u_host = oracle.uniforms(42, 3, B)
    d = lambda x: None if x is None else x.to(DEV)  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(d(w.logits), d(w.temperature), d(w.top_k), d(w.top_p), u_dev,
                           status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_sampler(w.logits, w.temperature, w.top_k, w.top_p, torch.from_numpy(u_host),
                  tok.cpu().numpy())
