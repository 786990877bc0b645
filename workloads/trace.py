"""Request arrivals for the continuous-batching trace.

Time is counted in scheduler steps.  At each step a Poisson(arrival_rate)
number of requests arrives; each has a log-normal prompt length (median
prompt_median, sigma prompt_sigma, rounded, clipped to [1, prompt_max]) and a
geometric output length on {1, 2, ...} with mean output_mean.  Request ids are
assigned in arrival order starting at 0.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .generators import SEED, _seed_list


@dataclass(frozen=True)
class Arrival:
    step: int
    req_id: int
    prompt_len: int
    max_output: int


def generate_arrivals(spec, name: str = "trace") -> list[Arrival]:
    rng = np.random.default_rng(_seed_list(SEED, name, "arrivals", spec.steps))
    out: list[Arrival] = []
    rid = 0
    for step in range(spec.steps):
        n = int(rng.poisson(spec.arrival_rate))
        for _ in range(n):
            p = float(rng.lognormal(np.log(spec.prompt_median), spec.prompt_sigma))
            prompt = int(min(max(round(p), 1), spec.prompt_max))
            output = int(rng.geometric(1.0 / spec.output_mean))
            out.append(Arrival(step, rid, prompt, output))
            rid += 1
    return out
