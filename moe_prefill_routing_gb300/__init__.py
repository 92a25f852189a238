"""GB300-native routed MoE prefill layer: plan -> gather -> grouped expert FFN -> combine.

Importing the package is cheap: the compiled library is loaded on the first
call through :mod:`moe_prefill_routing_gb300.binding`.
"""
__all__ = ["binding", "workload"]
