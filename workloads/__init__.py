"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark."""
from .gen import (CONFIGS, Workload, budget_sweep, dfly_block, greedy_mtp, random_case,
                  stochastic_mtp, tiny_chain, verify_cost_table)

__all__ = ["CONFIGS", "Workload", "budget_sweep", "dfly_block", "greedy_mtp", "random_case",
           "stochastic_mtp", "tiny_chain", "verify_cost_table"]
