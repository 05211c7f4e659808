"""Host plan: the decode given host copies of page_table_indptr and length_info
(desc->host_indptr / host_length_info) places its workers from them and reads the
sequences' lengths and page-table offsets from its launch.  The split and every
arithmetic step are the same as when it scans the device arrays, so the outputs must
be bitwise equal, and equal to the oracle within the usual tolerances."""
import numpy as np
import pytest
import torch

from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, gpu_decode, kind_of, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _meta(wl):
    return pd._lib.host_meta_of(wl.indptr, wl.length_info)


@pytest.mark.parametrize("name,over", [("llama3_8b_bf16", {}), ("window_sink_f16", {}),
                                       ("fp8_kv_highconc", {}), ("long_ctx_bf16", {}),
                                       ("tiny_fp32", {}), ("llama3_8b_bf16", dict(page_size=8, pool=1200)),
                                       ("llama3_8b_bf16", dict(rotary_mode=2))])
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_host_plan_is_bitwise_the_device_plan(name, over, splits):
    wl = W.make(name, seed=500 + splits, reduced=name != "tiny_fp32", **over).to(DEV)
    kw = dict(num_splits=splits)
    if splits > 1:
        kw["max_kv_len_hint"] = int(wl.attended.max())
    o1, l1 = gpu_decode(wl, **kw)
    o2, l2 = gpu_decode(wl, host_meta=_meta(wl), **kw)
    assert pd.check_device_errors() == "PD_OK"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    compare(kind_of(wl), o2, l2, ro, rl)


def test_host_plan_ignores_the_device_arrays():
    """With host copies the device indptr / length_info are not read: poisoning them
    changes nothing."""
    wl = W.make("llama3_8b_bf16", seed=510, reduced=True).to(DEV)
    meta = _meta(wl)
    o1, l1 = gpu_decode(wl, host_meta=meta)
    bad = W.Workload(**{**wl.__dict__, "indptr": torch.full_like(wl.indptr, 7),
                        "length_info": torch.full_like(wl.length_info, -3)})
    o2, l2 = gpu_decode(bad, host_meta=meta)
    assert pd.check_device_errors() == "PD_OK"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_plan_multi_query_and_edge_sequences():
    from tests.test_mq_gpu import _gpu, _mq, _oracle
    wl, Q = _mq("llama3_8b_bf16", 520, 3)
    meta = _meta(wl)
    o1, l1 = _gpu(wl, Q)
    o2, l2 = _gpu(wl, Q, host_meta=meta)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl, _ = _oracle(wl, Q, 3)
    compare("bf16", o2, l2, ro, rl)
    # empty, one-row and full-page sequences; an inconsistent window is reported as a
    # bad length by both plans alike
    from tests.test_decode_gpu import _custom
    e = _custom([0, 1, 16, 33, 0, 200], seed=3)
    o1, l1 = gpu_decode(e, num_splits=3)
    o2, l2 = gpu_decode(e, num_splits=3, host_meta=_meta(e))
    assert pd.check_device_errors() == "PD_OK"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_plan_too_large_falls_back_to_the_device_scan():
    # 1100 sequences do not fit the launch's 1024 ints: the device scan runs, same result
    wl = W.make("llama3_8b_bf16", seed=530, reduced=True, B=1100, len_dist=("uniform", 1, 40),
                pool=4000).to(DEV)
    o1, l1 = gpu_decode(wl)
    o2, l2 = gpu_decode(wl, host_meta=_meta(wl))
    assert pd.check_device_errors() == "PD_OK"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
