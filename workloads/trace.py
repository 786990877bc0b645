"""Request arrivals for the continuous-batching trace.

Time is counted in scheduler steps.  At each step a Poisson(arrival_rate)
number of requests arrives; each has a log-normal prompt length (median
prompt_median, sigma prompt_sigma, rounded, clipped to [1, prompt_max]) and a
geometric output length on {1, 2, ...} with mean output_mean.  Request ids are
assigned in arrival order starting at 0.

The prefix-sharing variant (`generate_prefix_arrivals`) gives every request
its prompt's token ids: most prompts start with one of a few shared system
prompts (popularity falling as 1/(k+1)), in one of two namespaces (standing
for two adapters or tenants), followed by a request-specific part; the rest
are unrelated prompts.  Token ids are uniform on [0, vocab).
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


@dataclass(frozen=True)
class PrefixArrival(Arrival):
    namespace: int = 0
    system: int = -1          # shared system prompt id, -1 if none
    system_len: int = 0       # the prompt's first system_len tokens are that system prompt
    tokens: tuple = ()        # the whole prompt's token ids


def generate_prefix_arrivals(spec, name: str = "prefix_trace", num_systems: int = 8,
                             system_median: int = 1536, user_median: int = 256,
                             share_prob: float = 0.75, other_namespace_prob: float = 0.15,
                             vocab: int = 32000) -> list[PrefixArrival]:
    rng = np.random.default_rng(_seed_list(SEED, name, "arrivals", spec.steps))
    limit = min(spec.prompt_max, spec.max_model_len - 1)
    systems = []
    for _ in range(num_systems):
        n = int(min(max(round(float(rng.lognormal(np.log(system_median), 0.5))), 16), limit // 2))
        systems.append(rng.integers(0, vocab, size=n, dtype=np.int64))
    weights = 1.0 / (np.arange(num_systems) + 1.0)
    weights /= weights.sum()
    out: list[PrefixArrival] = []
    rid = 0
    for step in range(spec.steps):
        for _ in range(int(rng.poisson(spec.arrival_rate))):
            output = int(rng.geometric(1.0 / spec.output_mean))
            if rng.random() < share_prob:
                k = int(rng.choice(num_systems, p=weights))
                ns = 1 if rng.random() < other_namespace_prob else 0
                u = int(min(max(round(float(rng.lognormal(np.log(user_median), 1.0))), 1),
                            limit - len(systems[k])))
                toks = np.concatenate([systems[k], rng.integers(0, vocab, size=u, dtype=np.int64)])
                sys_id, sys_len = k, len(systems[k])
            else:
                p = float(rng.lognormal(np.log(spec.prompt_median), spec.prompt_sigma))
                n = int(min(max(round(p), 1), limit))
                toks = rng.integers(0, vocab, size=n, dtype=np.int64)
                ns, sys_id, sys_len = 0, -1, 0
            out.append(PrefixArrival(step, rid, len(toks), output, ns, sys_id, sys_len,
                                     tuple(int(t) for t in toks)))
            rid += 1
    return out
