"""The benchmark's workloads and the arithmetic behind its numbers, pinned to
the sizes the walkthrough pages and the configuration table state (CPU only):
request counts, head groupings and lengths of each workload, the algorithmic
K/V bytes of the decode workloads, the causal flop count of the prefill
workload, and the whole-step floor that bench.py reports."""
import importlib.util
import os

import pytest

from paged_kv_attention_05_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_tiny_mixed_is_the_trace_of_the_tour():
    # "Tour: One forward pass", stop 3: 540 and 129 cached tokens decoding one
    # token each, a 298-token prompt; 304 rows with 4 padding slots
    s = W.spec("tiny_mixed")
    assert (s.num_reqs, s.hq, s.hkv) == (3, 32, 8)
    assert list(s.ctx) == [540, 129, 0] and list(s.q_len) == [1, 1, 298]
    assert s.num_tokens == 300 and s.pad_tokens == 4


def test_decode_workload_sizes():
    mha, gqa, mqa = W.spec("mha_decode"), W.spec("gqa_decode"), W.spec("mqa_long_decode")
    assert (mha.num_reqs, mha.hq, mha.hkv) == (256, 32, 32)
    assert set(mha.q_len) == {1} and 512 <= min(mha.ctx) and max(mha.ctx) <= 4096
    assert (gqa.num_reqs, gqa.hq, gqa.hkv) == (128, 32, 8) and set(gqa.ctx) == {8192}
    assert (mqa.num_reqs, mqa.hq, mqa.hkv) == (32, 32, 1) and set(mqa.ctx) == {32768}
    # K/V bytes read per step: (ctx + 1) keys x Hkv x 128 dims x 2 bytes x (K, V)
    assert gqa.kv_bytes() == 128 * 8193 * 8 * 128 * 2 * 2 == 4_295_491_584
    assert mqa.kv_bytes() == 32 * 32769 * 1 * 128 * 2 * 2 == 536_887_296
    assert mha.kv_bytes() == sum((c + 1) * 32 * 128 * 2 * 2 for c in mha.ctx)


def test_prefill_flops_and_bytes():
    s = W.spec("large_prefill")
    assert (s.num_reqs, s.hq, s.hkv) == (8, 64, 8)
    assert set(s.ctx) == {0} and set(s.q_len) == {2048}
    b = _bench()
    # 4 x 128 flops per (visible key, query row, query head), causal
    assert b.causal_flops(s) == 8 * 64 * 512 * 2048 * 2049 // 2 == 550_024_249_344
    # the whole step: K/V of every request read once + Q read + O written +
    # the write's new rows read (bf16) and stored
    kv = 8 * 2048 * 8 * 128 * 2 * 2
    qo = 2 * 16384 * 64 * 128 * 2
    wr = 16384 * 8 * 128 * 2 * (2 + 2)
    assert b.step_bytes(s) == kv + qo + wr


def test_mixed_chunked_composition():
    s = W.spec("mixed_chunked")
    chunks = [(c, n) for c, n in zip(s.ctx, s.q_len) if n > 1]
    decodes = [c for c, n in zip(s.ctx, s.q_len) if n == 1]
    assert sorted(chunks) == [(0, 224), (1024, 224)]
    assert len(decodes) == 64 and all(256 <= c <= 2048 for c in decodes)
    assert s.num_tokens == 512 and (s.hq, s.hkv) == (32, 8)


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_metric_units_and_floor(name):
    b = _bench()
    s = W.spec(name)
    metric, unit = b.metric_of(s)
    work = b.metric_work(s)
    if unit == "GB/s":
        assert work == pytest.approx(s.kv_bytes() / 1e9)
    elif unit == "TFLOP/s":
        assert work == pytest.approx(b.causal_flops(s) / 1e12)
    else:
        assert unit == "tokens/s" and work == s.num_tokens
    # the floor of a step: bytes over the copy rate or flops over the peak,
    # whichever is longer; decode steps are bound by bytes, the large prefill
    # by flops
    t_bytes = b.step_bytes(s) / 6765.3e9
    t_flops = b.causal_flops(s) / 1932.2e12
    if name in ("mha_decode", "gqa_decode", "mqa_long_decode"):
        assert t_bytes > t_flops
    if name == "large_prefill":
        assert t_flops > t_bytes


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
@pytest.mark.parametrize("elem", [2, 1])
def test_timed_steps_read_from_hbm(name, elem):
    # the timed loop rotates through enough copies of a step's inputs that the
    # rotation is at least four L2s, so no step finds its K/V still in L2
    b = _bench()
    sb = b.step_bytes(W.spec(name), elem)
    n = b.l2_copies(sb)
    assert n * sb >= 4 * 129e6 and (n == 1 or (n - 1) * sb < 4 * 129e6)
    if name in ("mha_decode", "gqa_decode", "large_prefill"):
        assert n == 1
    if name == "tiny_mixed":
        assert n > 40


def test_clock_record_takes_the_loaded_window(tmp_path):
    # nvidia-smi lines (timestamp first): one before the load, two inside it,
    # one of them with the power cap active; the record keeps the two
    import datetime
    import time
    b = _bench()
    now = time.time()

    def line(t, sm, cap):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return "%s, 0, %d, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, %s\n" % (
            ts, sm, "Active" if cap else "Not Active")

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    cs = b.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write(line(now - 1.0, 1200, False) + line(now + 0.1, 2070, True) +
                line(now + 0.3, 2040, False))
    cs.proc = Done()
    rec = cs.stop(now, now + 0.5)
    assert rec["samples"] == 2 and rec["sm_mhz"] == 2055.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["window"].startswith("the timed steps")


def test_decode_kernel_algorithmic_bytes():
    # every decode request's K/V rows once per KV head, its query row read and
    # output row written; prefill-class requests are not the decode kernel's
    b = _bench()
    assert b.decode_algorithmic_bytes(W.spec("gqa_decode")) == \
        4_295_491_584 + 128 * 2 * 32 * 128 * 2 == 4_297_588_736
    assert b.decode_algorithmic_bytes(W.spec("gqa_decode"), 1) == \
        4_295_491_584 // 2 + 128 * 2 * 32 * 128 * 2
    mqa = W.spec("mqa_long_decode")
    assert b.decode_algorithmic_bytes(mqa) == 536_887_296 + 32 * 2 * 32 * 128 * 2
    # the 512-token mixed batch: 64 decodes count, the two 224-token chunks do not
    mc = W.spec("mixed_chunked")
    dec = [(c, n) for c, n in zip(mc.ctx, mc.q_len) if n == 1]
    assert b.decode_algorithmic_bytes(mc) == sum(
        (c + 1) * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 for c, _ in dec)
    # a 3-token decode of a GQA group of 4 (12 rows) is decode work; 5 tokens are not
    s = W.custom([100, 100], [3, 5], 32, 8)
    assert b.decode_algorithmic_bytes(s) == 103 * 8 * 128 * 4 + 2 * 3 * 32 * 128 * 2
