"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark."""
from .gen import (CONFIGS, Workload, budget_sweep, dfly_block, greedy_mtp, random_case,
                  stochastic_mtp, tiny_chain)

__all__ = ["CONFIGS", "Workload", "budget_sweep", "dfly_block", "greedy_mtp", "random_case",
           "stochastic_mtp", "tiny_chain"]
