"""Static checks of the CUDA sources that need no GPU. Every mbarrier the
tcgen05 decode kernel waits on, commits to or arrives at is initialised (a
wait on an uninitialised barrier faults the context), and the barrier enum
gives every barrier its own 8-byte slot below kNumBars. Every spin-wait on a
barrier goes through the bounded waits."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "nvfp4_sparse_mla_gb300", "csrc")


def _source(name):
    with open(os.path.join(CSRC, name)) as f:
        src = f.read()
    # comments out: only code is checked
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def test_every_barrier_used_is_initialised():
    src = _source("decode_tc.cu")
    used = set(re.findall(r"\bbar\((kBar\w+)", src))
    inited = set(re.findall(r"mbar_init\(bar\((kBar\w+)", src))
    assert used, "no barrier uses found"
    assert used <= inited, f"waited on or signalled but never initialised: {sorted(used - inited)}"


def test_barrier_slots_are_distinct_and_dense():
    src = _source("decode_tc.cu") + _source("decode_tc_layout.h")
    body = re.search(r"enum Bar \{(.*?)\};", src, re.S).group(1)
    values = {n: int(v) for n, v in re.findall(r"(kBar\w+|kNumBars)\s*=\s*(\d+)", body)}
    n_bars = values.pop("kNumBars")
    # kBarPV + j for j < 4 (one per PV block of 128 value dims)
    width = {n: 1 for n in values}
    width["kBarPV"] = 4
    assert re.search(r"for \(int j = 0; j < 4; \+\+j\) mbar_init\(bar\(kBarPV \+ j\)", src)
    slots = sorted(s for n, v in values.items() for s in range(v, v + width[n]))
    assert slots == list(range(n_bars)), slots


def _body(src, signature):
    start = src.index(signature)
    return src[start:src.index("\n}", start) + 2]


def test_barrier_waits_are_bounded():
    src = _source("decode_tc.cu")
    # the raw try_wait sits only in the two single-shot helpers ...
    helpers = _body(src, "bool mbar_test(") + _body(src, "bool mbar_wait_hint(")
    assert src.count("mbarrier.try_wait") == helpers.count("mbarrier.try_wait") >= 2
    # ... which only the two bounded loops call, each with its time limit
    loops = [_body(src, "bool wait_bar("), _body(src, "void wait_bar_drain(")]
    for loop in loops:
        assert "globaltimer_ns()" in loop and "kWaitLimitNs" in loop
    for helper in ("mbar_test(", "mbar_wait_hint("):
        calls = src.count(helper) - 1  # less the definition
        assert calls == sum(loop.count(helper) for loop in loops) >= 1, helper
