"""Every stated round of the five workloads, library against the float64 oracle.

The rounds run from each workload's seed at its stated sizes and round count (1000 / 200 /
200 / 200 / 50); the oracle runs on all host cores (oracle.parallel).  Every output must match:
draft tokens, roots, branches, accept lengths, committed tokens, cache keys, hits and reuse
flags.  The float32 tier certifies its decisions and hands the rest to the float-float tier,
whose decisions are exact except within 2e-11 of a boundary (counted as unresolved); a
mismatch is allowed only at such a decision, and the stated budget caps mismatches at 1e-4 of
all decisions.  Runs for about two to four minutes on the GPU machine's host cores.
"""
import pytest

from oracle.parallel import OraclePool
from tests import sweep_rounds as SR

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    with OraclePool() as p:
        yield p


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_stated_rounds_match_the_oracle(pool, cfg):
    res = SR.sweep_config(cfg, SR.STATED[cfg], pool)
    g = res["gpu_stats"]
    unresolved = g.get("unresolved", 0) + g.get("sampler_unresolved", 0)
    assert res["sequences"] == SR.STATED[cfg] * SR.CONFIGS[cfg].B
    assert res["mismatches"] <= unresolved, res
    assert res["mismatches"] <= 1e-4 * res["decisions_oracle"], res
    if cfg == 4:
        assert res["root_logprob_max_abs_diff"] <= 1e-6, res
