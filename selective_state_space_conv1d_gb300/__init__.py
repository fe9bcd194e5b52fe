"""GB300-native Mamba-1 selective-SSM mixer core (placeholder until the binding lands)."""
