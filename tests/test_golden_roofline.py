"""The bench's roofline arithmetic against the worked examples the pages print
(tests/golden/roofline_examples.txt, each with its passage)."""
import os

import pytest

import bench

HERE = os.path.dirname(os.path.abspath(__file__))
FNS = {
    "read_bound": bench.read_bound_per_s,
    "fixed_cost": bench.fixed_cost_ms,
    "crossover": bench.compute_bound_concurrency,
    "matmul_tflops": bench.matmul_tflops,
}


def _examples():
    out = []
    with open(os.path.join(HERE, "golden", "roofline_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *vals = line.split()
            out.append((kind, [float(v) for v in vals[:-2]], float(vals[-2]), float(vals[-1])))
    return out


EXAMPLES = _examples()


def test_every_relation_has_an_example():
    assert {k for k, _, _, _ in EXAMPLES} == set(FNS)


@pytest.mark.parametrize("kind,args,printed,within", EXAMPLES)
def test_printed_example(kind, args, printed, within):
    got = FNS[kind](*args)
    assert abs(got - printed) <= within, (kind, args, got, printed)
