"""Writes rmsnorm_ties_27b_stack_m5.json: at each of the 129 RMSNorm sites of the oracle's own
64-layer pass over the 27B-shaped stack (M = 5, the bench's input rows), how the oracle's codes
(formed from x*w, reading R4) compare with the plain definition's (requantisation of (x*inv)*w).
Calls only the oracle and the seeded input generator.

    python tests/golden/make_rmsnorm_ties.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))          # tests/
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))  # repository root

import sdgen  # noqa: E402
from _rmsnorm_ties import TIE, compare_site, stack_sites  # noqa: E402


def main():
    spec = sdgen.StackSpec()
    sites = []
    for name, x, w in stack_sites(spec, 5, spec.layers):
        r = compare_site(x, w, sdgen.EPS)
        r["site"] = name
        sites.append(r)
        print(name, r, flush=True)
    codes = sum(s["codes"] for s in sites)
    diff = sum(s["differing"] for s in sites)
    out = {
        "what": "oracle RMSNorm codes (from x*w) vs the plain definition (requantised (x*inv)*w) at every norm "
                "site of the oracle's 64-layer pass, 27B-shaped 4-bit stack, M = 5, the bench's input rows",
        "tie_band": TIE,
        "sites": sites,
        "total_codes": codes,
        "total_differing": diff,
        "tie_rate": diff / codes,
    }
    with open(os.path.join(HERE, "rmsnorm_ties_27b_stack_m5.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(f"{diff} of {codes} codes differ ({diff / codes:.3e})")


if __name__ == "__main__":
    main()
