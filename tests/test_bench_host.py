"""Host logic of bench.py and of the workload table, on the CPU: the metric's
FLOP and byte counts against the figures the scope table prints for the five
configurations, the banded FLOP count against brute force, the reference
arm's row sampling against the full computation, and the rule that a DRAM
traffic record only counts while it describes the current kernel sources."""
import json
import os
import sys

import numpy as np
import pytest

import oracle
from exact_attention_82_gb300.inputs import WORKLOADS, Workload, make_qkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

BY_NAME = {w.name: w for w in WORKLOADS}


# The configurations' algorithmic FLOPs and bytes as printed in the scope
# table (metric: 4*B*H*Sq*Sk*D, halved when causal; Q, K, V read once, O and
# LSE written once), restated as integers.
@pytest.mark.parametrize("name,flops,nbytes", [
    ("b1h1s128d64", 4_194_304, 65_536 + 512),
    ("b8h16s2048d128", 274_877_906_944, 268_435_456 + 1_048_576),
    ("b4h16s4096d128_causal", 274_877_906_944, 268_435_456 + 1_048_576),
    ("b1h16s16384d128_causal", 1_099_511_627_776, 268_435_456 + 1_048_576),
    ("b16h32s1000d64_causal_q4", 65_536_000_000, 262_144_000 + 2_048_000),
])
def test_config_flops_and_bytes(name, flops, nbytes):
    w = BY_NAME[name]
    assert w.flops == flops
    assert w.hbm_bytes == nbytes


def _allowed_pairs(Sq, Sk, causal, wl):
    n = 0
    for i in range(Sq):
        for j in range(Sk):
            if causal and j > i:
                continue
            if wl >= 0 and j < i - wl:
                continue
            n += 1
    return n


@pytest.mark.parametrize("Sq,Sk,causal,wl", [(37, 37, True, 5), (64, 64, True, 0), (50, 80, False, 9),
                                             (33, 33, True, 100)])
def test_banded_flops_count_allowed_pairs(Sq, Sk, causal, wl):
    w = Workload("t", 2, 3, Sq, Sk, 16, causal, 1.0, wl)
    assert w.flops == 4.0 * 2 * 3 * 16 * _allowed_pairs(Sq, Sk, causal, wl)


def test_backward_and_fp8_counts():
    fwd, bwd, f8 = BY_NAME["b8h16s2048d128"], BY_NAME["b8h16s2048d128_bwd"], BY_NAME["b8h16s2048d128_fp8"]
    assert bwd.flops == 2.5 * fwd.flops          # five products against the forward's two
    assert f8.flops == fwd.flops
    # 1-byte Q, K, V; bf16 O and fp32 LSE as for 16-bit inputs
    assert f8.hbm_bytes == fwd.hbm_bytes - 8 * 16 * (3 * 2048 * 128)


def test_source_groups():
    assert bench.source_group("fwd") == bench.source_group("fp8") == "fwd"
    assert bench.source_group("bwd") == "bwd" and bench.source_group("splitkv") == "splitkv"
    for g in ("fwd", "bwd", "splitkv"):
        for rel in bench.KERNEL_SOURCES[g]:
            assert os.path.exists(os.path.join(ROOT, rel)), rel


def test_traffic_record_needs_current_sources(tmp_path, monkeypatch):
    w = BY_NAME["b8h16s2048d128"]
    rec = {w.name: {"kernel_group": "fwd", "kernel_sha256": bench.kernel_source_hash("fwd"),
                    "dram_bytes_per_launch": 123}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_per_launch(w) == 123
    rec[w.name]["kernel_sha256"] = "0" * 64          # taken on other sources
    f.write_text(json.dumps(rec))
    assert bench.traffic_per_launch(w) is None
    assert bench.traffic_per_launch(BY_NAME["b1h1s128d64"]) is None   # never captured
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.traffic_per_launch(w) is None


def test_source_key_ignores_comments_but_not_code():
    """The key of a DRAM record survives comment edits but not code edits."""
    base = 'int f(int x) { return x + 1; }  // add one\nconst char *s = "// kept";\n'
    same = '/* header */\nint f(int x) { return x + 1; }\n\nconst char *s = "// kept"; // note\n'
    code = 'int f(int x) { return x + 2; }  // add one\nconst char *s = "// kept";\n'
    lit = 'int f(int x) { return x + 1; }  // add one\nconst char *s = "// kapt";\n'
    k = bench._strip_comments
    assert k(base) == k(same)
    assert k(base) != k(code) and k(base) != k(lit)
    assert '"// kept"' in k(base)


@pytest.mark.parametrize("causal,wl,r0,rows", [(True, 40, 50, 30), (True, -1, 10, 20), (False, -1, 64, 7),
                                               (True, 8, 0, 16)])
def test_reference_sampler_rows_equal_full_computation(monkeypatch, causal, wl, r0, rows):
    """The reference arm evaluates a block of query rows on exactly the keys they
    may see, with the band re-expressed in the slice's indices; its output must
    be those rows of the full computation, and its FLOP count theirs."""
    B, H, S, D = 1, 2, 96, 16
    w = Workload("t", B, H, S, S, D, causal, 1.0, wl)
    q, k, v = make_qkv(B, H, S, S, D, seed=31)
    sampler = bench._RowSampler(w, q, k, v, None, nh=H)
    got = {}
    real = oracle.attn_fwd

    def spy(*a, **kw):
        got["out"] = real(*a, **kw)
        return got["out"]

    monkeypatch.setattr(oracle, "attn_fwd", spy)
    _, flops = sampler.run(r0, rows)
    o_full, l_full = real(sampler.q[None], sampler.k[None], sampler.v[None], w.scale, False, w.window)
    o_s, l_s = got["out"]
    r1 = min(S, r0 + rows)
    np.testing.assert_allclose(o_s[0], o_full[0][:, r0:r1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l_s[0], l_full[0][:, r0:r1], rtol=1e-12, atol=1e-13)
    pairs = sum(1 for i in range(r0, r1) for j in range(S)
                if not (causal and j > i) and not (wl >= 0 and j < i - wl))
    assert flops == 4.0 * D * pairs * H


@pytest.mark.parametrize("S,stride,causal", [(300, 2, True), (520, 3, False), (128, 2, True), (1, 2, False)])
def test_blockmask_flops_count_allowed_pairs(S, stride, causal):
    """The block-mask workloads' FLOPs: 4*B*H*D times the allowed pairs, counted here
    by brute force over every (query, key) pair of the pattern."""
    from exact_attention_82_gb300.inputs import dilated_block_mask

    w = Workload("t", 2, 3, S, S, 16, causal, path="blockmask", dilation=stride)
    m = dilated_block_mask(-(-S // 128), -(-S // 128), stride, causal)[0].numpy()
    pairs = sum(1 for i in range(S) for j in range(S) if m[i // 128, j // 128] and not (causal and j > i))
    assert w.flops == 4.0 * 2 * 3 * 16 * pairs
    assert w.hbm_bytes == 2 * 3 * (2 * 3 * S * 16 + 2 * S * 16 + 4 * S) + m.size


@pytest.mark.parametrize("causal,r0,rows", [(True, 130, 100), (False, 0, 128), (True, 0, 300)])
def test_reference_sampler_blockmask_rows_equal_full_computation(monkeypatch, causal, r0, rows):
    """For a block mask the reference arm evaluates whole query blocks against
    every key, the causal bound shifted to the slice; its output must be those rows
    of the full computation, and its FLOP count theirs."""
    B, H, S, D = 1, 2, 300, 16
    w = Workload("t", B, H, S, S, D, causal, path="blockmask", dilation=2)
    q, k, v = make_qkv(B, H, S, S, D, seed=32)
    sampler = bench._RowSampler(w, q, k, v, None, nh=H)
    got = {}
    real = oracle.attn_fwd_blockmask

    def spy(*a, **kw):
        got["out"] = real(*a, **kw)
        return got["out"]

    monkeypatch.setattr(oracle, "attn_fwd_blockmask", spy)
    _, flops = sampler.run(r0, rows)
    o_full, l_full = real(sampler.q[None], sampler.k[None], sampler.v[None], w.scale, w.block_mask.numpy(),
                          window=w.window, block=(128, 128))
    rb0, rb1 = (r0 // 128) * 128, min(S, -(-(r0 + rows) // 128) * 128)
    o_s, l_s = got["out"]
    np.testing.assert_allclose(o_s[0], o_full[0][:, rb0:rb1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l_s[0], l_full[0][:, rb0:rb1], rtol=1e-12, atol=1e-13)
    m = w.block_mask[0].numpy()
    pairs = sum(1 for i in range(rb0, rb1) for j in range(S) if m[i // 128, j // 128] and not (causal and j > i))
    assert flops == 4.0 * D * pairs * H
