"""Device-side failure detection without a GPU fault: a bounded wait that nothing
satisfies gives up, the status word says so, and the context stays usable."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    import sparse_attention_serving_gb300 as dsa
    from gpu_helpers import bf, i32, to_u16
    from workloads import CONFIGS, prefill
    cfg = CONFIGS["tiny128"]
    ws = dsa.new_workspace(max(4096, dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, cfg.B, cfg.T, cfg.T,
                                                         cfg.H_I, cfg.topk)))
    code, where, detail = dsa.selftest_wait_timeout(ws, 20_000_000)
    assert code == dsa.DSA_ERR_DEVICE_TIMEOUT and where == 0x500
    assert dsa.read_device_status(ws)[0] == dsa.DSA_OK  # reading clears it
    # the context is still usable: a real call afterwards succeeds
    d = prefill(cfg)
    idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_idx"])),
                               i32(d["q_start"]), i32(d["kv_len"]), cfg.topk, cfg.T, workspace=ws)
    torch.cuda.synchronize()
    assert dsa.read_device_status(ws)[0] == dsa.DSA_OK
    gi = idx.cpu().numpy()[0]
    assert all(sorted(gi[t, :t + 1].tolist()) == list(range(t + 1)) for t in range(cfg.T))


def test_selftest_rejects_long_limits():
    import sparse_attention_serving_gb300 as dsa
    ws = dsa.new_workspace(4096)
    with pytest.raises(dsa.DsaError):
        dsa.selftest_wait_timeout(ws, 10_000_000_000)


def test_prefill_indexer_workspace_too_small_is_rejected():
    """The prefill indexer's candidate buffers live in the workspace: a workspace
    smaller than dsa_workspace_bytes reports is rejected before any launch."""
    import sparse_attention_serving_gb300 as dsa
    from gpu_helpers import bf, i32
    from workloads import CONFIGS, prefill
    cfg = CONFIGS["tiny128"]
    d = prefill(cfg)
    need = dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, cfg.B, cfg.T, cfg.T, cfg.H_I, cfg.topk)
    ws = dsa.new_workspace(need - 256)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_idx"])),
                             i32(d["q_start"]), i32(d["kv_len"]), cfg.topk, cfg.T, workspace=ws)
    assert e.value.code == dsa.DSA_ERR_WORKSPACE_TOO_SMALL
